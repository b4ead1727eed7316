"""Pins of the oracle's LM-head product (logits = hidden x weight^T from bf16
inputs, in double precision): a brute-force sum, one-hot rows, known bf16 bit
patterns and the error scale it reports."""
import numpy as np

import oracle
import workloads


def test_matches_a_brute_force_sum():
    h, w, _ = workloads.lm_head(61, 3, 17, 70)
    L, A = oracle.lm_head_logits(h, w)
    hf = workloads.bf16_bits_to_f32(h).reshape(3, 70)
    wf = workloads.bf16_bits_to_f32(w).reshape(17, 70)
    for i in range(3):
        for v in range(17):
            s, a = 0.0, 0.0
            for k in range(70):
                s += float(hf[i, k]) * float(wf[v, k])
                a += abs(float(hf[i, k]) * float(wf[v, k]))
            assert abs(L[i, v] - s) <= 1e-12 * a
            assert abs(A[i, v] - a) <= 1e-12 * a


def test_one_hot_rows_pick_weight_columns():
    _, w, _ = workloads.lm_head(62, 2, 40, 96)
    h = np.zeros((3, 96), np.uint16)
    h[0, 5] = 0x3F80   # 1.0
    h[1, 95] = 0xC000  # -2.0
    h[2, 0] = 0x3F81   # 1 + 2^-7
    L, _ = oracle.lm_head_logits(h, w)
    col = workloads.bf16_bits_to_f32(w).reshape(40, 96).astype(np.float64)
    assert np.array_equal(L[0], col[:, 5])
    assert np.array_equal(L[1], -2.0 * col[:, 95])
    assert np.array_equal(L[2], (1.0 + 2.0 ** -7) * col[:, 0])


def test_selected_columns_and_error_scale():
    h, w, _ = workloads.lm_head(63, 4, 300, 128)
    L, A = oracle.lm_head_logits(h, w)
    cols = np.array([299, 0, 150, 7])
    Ls, As = oracle.lm_head_logits(h, w, cols)
    assert np.array_equal(Ls, L[:, cols]) and np.array_equal(As, A[:, cols])
    assert np.all(A >= np.abs(L))
    assert 1.0 < L.std() < 3.0  # the workload's logits are ~ N(0, 4)
