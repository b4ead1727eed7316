// philox.cuh -- counter-based noise for the Gumbel-max pick.
//
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy
// as 1, 2, 3", SC'11): ten rounds; each round takes the 32x32->64 products of
// counter lanes 0 and 2 with the two Philox multipliers, crosses the high halves
// into lanes 0 / 2 xored with lanes 1 / 3 and the round key, and moves the low
// halves to lanes 1 / 3. The key advances by the two Weyl constants per round.
//
// Noise layout of the sampler (shared definition with its users, see sampler.h):
// token v of a row draws word (v & 3) of the block at counter
// (v >> 2, stream, offset_lo, offset_hi) under the row's 64-bit key.
#pragma once

#include <cstdint>

namespace dst {

struct PhiloxKey {
    uint32_t lo, hi;
};

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, PhiloxKey k)
{
    constexpr uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;
    constexpr uint32_t kWeylA = 0x9E3779B9u, kWeylB = 0xBB67AE85u;
    uint32_t k0 = k.lo, k1 = k.hi;
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t hiA = __umulhi(kMulA, c.x), loA = kMulA * c.x;
        const uint32_t hiB = __umulhi(kMulB, c.z), loB = kMulB * c.z;
        c = make_uint4(hiB ^ c.y ^ k0, loB, hiA ^ c.w ^ k1, loA);
        k0 += kWeylA;
        k1 += kWeylB;
    }
    return c;
}

// The 32x32 -> 64 product of the two Philox lanes in one instruction.
__device__ __forceinline__ void mul_wide(uint32_t a, uint32_t b, uint32_t& hi, uint32_t& lo)
{
    unsigned long long r;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(r) : "r"(a), "r"(b));
    lo = uint32_t(r);
    hi = uint32_t(r >> 32);
}

// Philox4x32-10 for the counters (b, c1, c2, c3) of one row, where only b varies:
// the first round's product of counter lane 2 and the second round's product of
// counter lane 0 depend on the row alone, so they are taken once per row. Same
// output as philox4x32_10(make_uint4(b, c1, c2, c3), key).
struct RowPhilox {
    uint32_t k0[10], k1[10];  // round keys (entries 0 and 1 unused after folding)
    uint32_t r1z;             // round 1: lane 3 of the counter xor round key 1
    uint32_t r2x;             // round 2: what lane 0 takes besides the varying product
    uint32_t r2z;             // round 2: lane 2 is r2z xor the round-1 low product
    uint32_t r2w;             // round 2 output lane 3 (a row constant)
};

__device__ __forceinline__ RowPhilox row_philox(PhiloxKey k, uint32_t c1, uint32_t c2, uint32_t c3)
{
    constexpr uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;
    RowPhilox p;
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        p.k0[round] = k.lo + uint32_t(round) * 0x9E3779B9u;
        p.k1[round] = k.hi + uint32_t(round) * 0xBB67AE85u;
    }
    uint32_t hb, lb, ha, la;
    mul_wide(kMulB, c2, hb, lb);            // round 1, lane 2: a row constant
    const uint32_t x1 = hb ^ c1 ^ p.k0[0];  // round 1 output lane 0
    p.r1z = c3 ^ p.k1[0];
    mul_wide(kMulA, x1, ha, la);            // round 2, lane 0: a row constant
    p.r2x = lb ^ p.k0[1];
    p.r2z = ha ^ p.k1[1];
    p.r2w = la;
    return p;
}

__device__ __forceinline__ uint4 philox_block(const RowPhilox& p, uint32_t b)
{
    constexpr uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;
    uint32_t ha, la, hb, lb;
    mul_wide(kMulA, b, ha, la);                 // round 1, lane 0
    mul_wide(kMulB, ha ^ p.r1z, hb, lb);        // round 2, lane 2
    uint32_t x = hb ^ p.r2x, y = lb, z = p.r2z ^ la, w = p.r2w;
#pragma unroll
    for (int round = 2; round < 10; ++round) {
        mul_wide(kMulA, x, ha, la);
        mul_wide(kMulB, z, hb, lb);
        const uint32_t nx = hb ^ y ^ p.k0[round], nz = ha ^ w ^ p.k1[round];
        x = nx;
        y = lb;
        z = nz;
        w = la;
    }
    return make_uint4(x, y, z, w);
}

__device__ __forceinline__ uint32_t lane_of(uint4 b, uint32_t i)
{
    return i == 0 ? b.x : (i == 1 ? b.y : (i == 2 ? b.z : b.w));
}

// u = (2 * (w >> 9) + 1) * 2^-24, exactly, in fp32: 1 + m * 2^-23 minus (1 - 2^-24).
__device__ __forceinline__ float noise_u(uint32_t w)
{
    return __uint_as_float(0x3F800000u | (w >> 9)) - 0x1.fffffep-1f;
}

// 1 - u, exactly: the same construction on the complemented word.
__device__ __forceinline__ float noise_one_minus_u(uint32_t w)
{
    return __uint_as_float(0x3F800000u | ((~w) >> 9)) - 0x1.fffffep-1f;
}

// E = -ln(u) in fp32, accurate near u = 1 through log1p of the exact 1 - u.
__device__ __forceinline__ float noise_exp1_f32(uint32_t w)
{
    const float u = noise_u(w);
    return (u <= 0.5f) ? -logf(u) : -log1pf(-noise_one_minus_u(w));
}

// The same draw in double precision (used to settle the final comparison).
__device__ __forceinline__ double noise_exp1_f64(uint32_t w)
{
    const double u = (2.0 * double(w >> 9) + 1.0) * 0x1p-24;
    return -log(u);
}

}  // namespace dst
