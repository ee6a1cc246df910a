// pkv_quant.cuh -- the K8/V4 quantisation of one (token, kv head) row by one
// warp, shared by the write kernel and the fused decode step so that both
// produce the same codes and scales bit for bit.
// [metalworking "The KV Cache", §"The K/V asymmetry": K stays at 8 bits, V goes
//  to 4; MTPLX "How MTPLX Manages Memory with KV Caching Strategies", the
//  quantised write path with per-block scale and zero tensors.]
// The fp32 operation sequence is fixed: IEEE division (__fdiv_rn), IEEE
// subtraction (__fsub_rn, never contracted), round-half-even (rintf), and RNE
// conversion of scales to fp16 before they are used.
#pragma once

#include "pkv_device.cuh"

namespace pkv {

// This lane's share of a quantised row: dims [lane*E, lane*E + E), E = D/32.
template <int D>
struct QuantRow {
    static constexpr int E = D / 32;
    uint32_t kpack;   // E int8 codes, dim lane*E in the low byte
    uint32_t vpack;   // E 4-bit codes, even dim in the low nibble
    __half ks;        // the row's K scale (the same in every lane)
    __half vs, vz;    // V scale and zero of this lane's 32-dim group
};

// kb / vb: this lane's E source values (fp16 or bf16 bits).
template <typename Src, int D>
__device__ __forceinline__ QuantRow<D> quantize_vals(const uint16_t (&kb)[D / 32], const uint16_t (&vb)[D / 32]) {
    constexpr int E = D / 32;
    constexpr int LPG = 32 / E;   // lanes per 32-dim V group
    QuantRow<D> r;
    float k[E], v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
        k[e] = Half16<Src>::to_float(kb[e]);
        v[e] = Half16<Src>::to_float(vb[e]);
    }
    // K: symmetric int8, one fp16 scale per (token, kv head)
    float a = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) a = fmaxf(a, fabsf(k[e]));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    r.ks = __float2half_rn(__fdiv_rn(a, 127.0f));
    const float s = __half2float(r.ks);
    r.kpack = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float c = (s == 0.f) ? 0.f : fminf(fmaxf(rintf(__fdiv_rn(k[e], s)), -127.f), 127.f);
        r.kpack |= (uint32_t(int32_t(c)) & 0xffu) << (8 * e);
    }
    // V: asymmetric 4-bit per group of 32 dims, fp16 scale and fp16 zero per group
    float lo = v[0], hi = v[0];
#pragma unroll
    for (int e = 1; e < E; ++e) {
        lo = fminf(lo, v[e]);
        hi = fmaxf(hi, v[e]);
    }
#pragma unroll
    for (int o = LPG / 2; o >= 1; o >>= 1) {
        lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lo == 0.f) lo = 0.f;  // a zero minimum is stored as +0
    r.vs = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), 15.0f));
    r.vz = __float2half_rn(lo);
    const float vs = __half2float(r.vs), vz = __half2float(r.vz);
    r.vpack = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const float c = (vs == 0.f) ? 0.f : fminf(fmaxf(rintf(__fdiv_rn(__fsub_rn(v[e], vz), vs)), 0.f), 15.f);
        r.vpack |= uint32_t(c) << (4 * e);
    }
    return r;
}

// ksrc / vsrc point at this lane's E source values (fp16 or bf16 bits).
template <typename Src, int D>
__device__ __forceinline__ QuantRow<D> quantize_row(const uint16_t* ksrc, const uint16_t* vsrc) {
    uint16_t kb[D / 32], vb[D / 32];
#pragma unroll
    for (int e = 0; e < D / 32; ++e) {
        kb[e] = ksrc[e];
        vb[e] = vsrc[e];
    }
    return quantize_vals<Src, D>(kb, vb);
}

}  // namespace pkv
