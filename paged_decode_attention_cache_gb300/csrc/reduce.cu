// reduce.cu -- split-KV phase 2: log-sum-exp combination of partition partials.
//
// The pages name split-KV decode [mlxcel manual "KV Cache", §"Paged Decode
// Storage and Kernels": decode splits; metalworking "The KV Cache": split-KV
// decode kernels] without printing the combination; this is the exact identity
//   M = max_p m_p,  w_p = l_p exp(m_p - M),  out = sum_p w_p o_p / sum_p w_p
// under which split attention equals single-pass attention.  Partitions with
// l_p = 0 (no visible token for that row) carry no weight.
//
// One warp per (row, head): lanes take 32 partitions at a time, compute their
// weights, and broadcast them by shuffle while every lane accumulates its
// head_dim/32 output dims (coalesced 128-bit or 64-bit loads of o_p).
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kWarps = 4;

template <int D>
__global__ void __launch_bounds__(kWarps * 32) lse_reduce_kernel(ReduceParams p) {
    constexpr int DPL = D / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = blockIdx.x;
    const int s = r / p.q_len;
    int ctx = p.context_lens[s];
    if (ctx < 0) ctx = 0;
    int nparts = (ctx + p.partition_size - 1) / p.partition_size;
    if (nparts > p.max_partitions) nparts = p.max_partitions;
    for (int h = blockIdx.y * kWarps + warp; h < p.num_heads; h += gridDim.y * kWarps) {
        const size_t base = (size_t(r) * p.num_heads + h) * p.max_partitions;
        // pass 1: global max over partitions with weight
        float M = -INFINITY;
        for (int i = lane; i < nparts; i += 32)
            if (p.exp_sums[base + i] > 0.f) M = fmaxf(M, p.max_logits[base + i]);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float acc[DPL];
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[e] = 0.f;
        float W = 0.f;
        if (M != -INFINITY) {
            for (int c0 = 0; c0 < nparts; c0 += 32) {
                const int i = c0 + lane;
                float w = 0.f;
                if (i < nparts) {
                    const float l = p.exp_sums[base + i];
                    if (l > 0.f) w = l * exp2f((p.max_logits[base + i] - M) * kLog2e);
                }
                W += w;
                const int n = min(32, nparts - c0);
                for (int k = 0; k < n; ++k) {
                    const float wk = __shfl_sync(0xffffffffu, w, k);
                    if (wk == 0.f) continue;
                    const float* o = p.tmp_out + (base + c0 + k) * D + lane * DPL;
                    if constexpr (DPL == 4) {
                        const float4 v = *reinterpret_cast<const float4*>(o);
                        acc[0] = fmaf(wk, v.x, acc[0]);
                        acc[1] = fmaf(wk, v.y, acc[1]);
                        acc[2] = fmaf(wk, v.z, acc[2]);
                        acc[3] = fmaf(wk, v.w, acc[3]);
                    } else {
                        const float2 v = *reinterpret_cast<const float2*>(o);
                        acc[0] = fmaf(wk, v.x, acc[0]);
                        acc[1] = fmaf(wk, v.y, acc[1]);
                    }
                }
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
        }
        const float inv = (W > 0.f) ? 1.f / W : 0.f;
        const size_t ob = (size_t(r) * p.num_heads + h) * D + lane * DPL;
#pragma unroll
        for (int e = 0; e < DPL; ++e) store_out(p.out, p.out_dtype, ob + e, acc[e] * inv);
    }
}

}  // namespace

cudaError_t launch_reduce(const ReduceParams& p, cudaStream_t stream) {
    const int rows = p.num_seqs * p.q_len;
    int hy = (p.num_heads + kWarps - 1) / kWarps;
    if (hy > 65535) hy = 65535;
    dim3 grid(rows, hy);
    if (p.head_dim == 128)
        lse_reduce_kernel<128><<<grid, kWarps * 32, 0, stream>>>(p);
    else
        lse_reduce_kernel<64><<<grid, kWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pkv
