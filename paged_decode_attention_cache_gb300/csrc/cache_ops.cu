// cache_ops.cu -- writes into and reads out of the paged cache:
//   reshape_and_cache  scatter new K/V rows into their slots (bit-exact copy)
//   gather_kv_cache    copy each sequence's visible tokens back to contiguous rows
//   quantize_kv        K int8 symmetric + V 4-bit asymmetric write path
// All three are pure data movement bounded by HBM: 16-byte vector accesses,
// consecutive threads on consecutive 16-byte chunks of a token row.
#include <type_traits>

#include "pkv_device.cuh"
#include "pkv_quant.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kBlockSize = 16;
constexpr int kThreads = 256;

// ---------------------------------------------------------------- reshape_and_cache
// [mlxcel manual "KV Cache", §"Attention Dispatch and In-Place Decode Writes":
//  the new row is written straight into the cache buffer; metalworking "The KV
//  Cache" names the reshape_and_cache kernel.]  One token's K (or V) row across
// all kv heads is contiguous in both the source [T, Hkv, D] and the cache
// [NB, 16, Hkv, D], so each token is `chunks` 16-byte chunks copied verbatim.
__global__ void __launch_bounds__(kThreads) reshape_and_cache_kernel(CacheWriteParams p, int chunks) {
    grid_dep_wait();
    grid_dep_launch();
    const int64_t total = int64_t(p.num_tokens) * chunks;
    const int64_t pool = int64_t(p.num_blocks) * kBlockSize;
    for (int64_t i = blockIdx.x * int64_t(kThreads) + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * kThreads) {
        const int64_t tok = i / chunks;
        const int c = int(i - tok * chunks);
        const int64_t slot = p.slot_mapping[tok];
        if (slot < 0) continue;  // padding
        if (slot >= pool) {
            if (c == 0) flag_error(p.err, PKV_DEVERR_OOB_SLOT);
            continue;
        }
        const uint4* ks = reinterpret_cast<const uint4*>(p.k_new) + tok * chunks + c;
        const uint4* vs = reinterpret_cast<const uint4*>(p.v_new) + tok * chunks + c;
        uint4* kd = reinterpret_cast<uint4*>(p.k_cache) + slot * chunks + c;
        uint4* vd = reinterpret_cast<uint4*>(p.v_cache) + slot * chunks + c;
        *kd = __ldg(ks);
        *vd = __ldg(vs);
    }
}

// ---------------------------------------------------------------- gather_kv_cache
// [metalworking "The KV Cache": fixed-size blocks plus an indirection table;
//  gather_kv_cache names the read back to contiguous storage.]  CTA (b, s)
// copies logical block b of sequence s.
__global__ void __launch_bounds__(kThreads) gather_kernel(GatherParams p, int chunks) {
    grid_dep_wait();
    grid_dep_launch();
    const int s = blockIdx.y, b = blockIdx.x;
    int ctx = p.context_lens[s];
    const int cap = p.max_blocks * kBlockSize;
    if (ctx > cap) {
        if (b == 0 && threadIdx.x == 0) flag_error(p.err, PKV_DEVERR_CAPACITY);
        ctx = cap;
    }
    const int t0 = b * kBlockSize;
    if (t0 >= ctx) return;
    const int ntok = min(kBlockSize, ctx - t0);
    const int pb = p.block_tables[int64_t(s) * p.max_blocks + b];
    if (pb < 0 || pb >= p.num_blocks) {
        if (threadIdx.x == 0) flag_error(p.err, PKV_DEVERR_OOB_BLOCK);
        return;
    }
    const int64_t dst_row0 = int64_t(p.cu_seq_lens[s]) + t0;
    const uint4* ksrc = reinterpret_cast<const uint4*>(p.k_cache) + int64_t(pb) * kBlockSize * chunks;
    const uint4* vsrc = reinterpret_cast<const uint4*>(p.v_cache) + int64_t(pb) * kBlockSize * chunks;
    uint4* kdst = reinterpret_cast<uint4*>(p.k_out) + dst_row0 * chunks;
    uint4* vdst = reinterpret_cast<uint4*>(p.v_out) + dst_row0 * chunks;
    const int n = ntok * chunks;  // the block's first ntok token rows are contiguous
    for (int i = threadIdx.x; i < n; i += kThreads) {
        kdst[i] = __ldg(ksrc + i);
        vdst[i] = __ldg(vsrc + i);
    }
}

// ---------------------------------------------------------------- dequantising gather
// [metalworking "The KV Cache", §"The K/V asymmetry": k = c * s, v = c * s + z;
//  gather as above.]  CTA (b, s) expands logical block b of sequence s; a
// thread takes 8 dims of one (token, kv head): one 8-byte K load, one 4-byte V
// load, two 16-byte stores.
template <typename OutT, int D>
__global__ void __launch_bounds__(kThreads) gather_dequant_kernel(GatherParams p) {
    grid_dep_wait();
    grid_dep_launch();
    constexpr int NG = D / 32;
    constexpr int CPT = D / 8;   // 8-dim chunks per (token, kv head)
    const int s = blockIdx.y, b = blockIdx.x;
    int ctx = p.context_lens[s];
    const int cap = p.max_blocks * kBlockSize;
    if (ctx > cap) {
        if (b == 0 && threadIdx.x == 0) flag_error(p.err, PKV_DEVERR_CAPACITY);
        ctx = cap;
    }
    const int t0 = b * kBlockSize;
    if (t0 >= ctx) return;
    const int ntok = min(kBlockSize, ctx - t0);
    const int pb = p.block_tables[int64_t(s) * p.max_blocks + b];
    if (pb < 0 || pb >= p.num_blocks) {
        if (threadIdx.x == 0) flag_error(p.err, PKV_DEVERR_OOB_BLOCK);
        return;
    }
    const int H = p.num_kv_heads;
    const int64_t dst_row0 = int64_t(p.cu_seq_lens[s]) + t0;
    const int n = ntok * H * CPT;
    for (int i = threadIdx.x; i < n; i += kThreads) {
        const int c = i % CPT, th = i / CPT, h = th % H, tt = th / H;
        const int64_t row = (int64_t(pb) * kBlockSize + tt) * H + h;          // cache row
        const int64_t meta = (int64_t(pb) * H + h) * kBlockSize + tt;           // scale index
        const uint2 kc = __ldg(reinterpret_cast<const uint2*>(static_cast<const int8_t*>(p.k_cache) + row * D) + c);
        const uint32_t vc = __ldg(reinterpret_cast<const uint32_t*>(static_cast<const uint8_t*>(p.v_cache) + row * (D / 2)) + c);
        const float ks = __half2float(__ldg(static_cast<const __half*>(p.k_scale) + meta));
        const float vs = __half2float(__ldg(static_cast<const __half*>(p.v_scale) + meta * NG + c / 4));
        const float vz = __half2float(__ldg(static_cast<const __half*>(p.v_zero) + meta * NG + c / 4));
        float kv[8], vv[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t kw = e < 4 ? kc.x : kc.y;
            const int code = int(int8_t((kw >> (8 * (e & 3))) & 0xffu));
            kv[e] = float(code) * ks;                                   // exact
            vv[e] = fmaf(float((vc >> (4 * e)) & 0xfu), vs, vz);        // one rounding
        }
        uint4 ko, vo;
        uint32_t* kw = &ko.x;
        uint32_t* vw = &vo.x;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if constexpr (sizeof(OutT) == 2 && std::is_same<OutT, __nv_bfloat16>::value) {
                const __nv_bfloat162 a = __floats2bfloat162_rn(kv[2 * e], kv[2 * e + 1]);
                const __nv_bfloat162 z = __floats2bfloat162_rn(vv[2 * e], vv[2 * e + 1]);
                memcpy(kw + e, &a, 4);
                memcpy(vw + e, &z, 4);
            } else {
                const __half2 a = __floats2half2_rn(kv[2 * e], kv[2 * e + 1]);
                const __half2 z = __floats2half2_rn(vv[2 * e], vv[2 * e + 1]);
                memcpy(kw + e, &a, 4);
                memcpy(vw + e, &z, 4);
            }
        }
        const int64_t dst = ((dst_row0 + tt) * H + h) * D + 8 * c;
        *reinterpret_cast<uint4*>(static_cast<OutT*>(p.k_out) + dst) = ko;
        *reinterpret_cast<uint4*>(static_cast<OutT*>(p.v_out) + dst) = vo;
    }
}

// ---------------------------------------------------------------- quantize_kv
// One warp per (token, kv head); the arithmetic is quantize_row (pkv_quant.cuh).
template <typename Src, int D>
__global__ void __launch_bounds__(kThreads) quantize_kernel(CacheWriteParams p) {
    grid_dep_wait();
    grid_dep_launch();
    constexpr int E = D / 32;            // values per lane
    constexpr int NG = D / 32;           // V groups per row
    constexpr int LPG = 32 / E;          // lanes per group
    const int lane = threadIdx.x & 31;
    const int64_t w = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int H = p.num_kv_heads;
    if (w >= int64_t(p.num_tokens) * H) return;
    const int64_t tok = w / H;
    const int h = int(w - tok * H);
    const int64_t slot = p.slot_mapping[tok];
    if (slot < 0) return;
    if (slot >= int64_t(p.num_blocks) * kBlockSize) {
        if (lane == 0) flag_error(p.err, PKV_DEVERR_OOB_SLOT);
        return;
    }
    const int64_t blk = slot / kBlockSize;
    const int off = int(slot - blk * kBlockSize);
    const int64_t src = (tok * H + h) * D + lane * E;
    const QuantRow<D> q = quantize_row<Src, D>(reinterpret_cast<const uint16_t*>(p.k_new) + src,
                                               reinterpret_cast<const uint16_t*>(p.v_new) + src);
    const int64_t row = (blk * kBlockSize + off) * H + h;
    const int64_t meta = (blk * H + h) * kBlockSize + off;
    int8_t* kq = reinterpret_cast<int8_t*>(p.k_cache) + row * D + lane * E;
    if constexpr (E == 4)
        *reinterpret_cast<uint32_t*>(kq) = q.kpack;
    else
        *reinterpret_cast<uint16_t*>(kq) = uint16_t(q.kpack);
    if (lane == 0) reinterpret_cast<__half*>(p.k_scale)[meta] = q.ks;
    uint8_t* vq = reinterpret_cast<uint8_t*>(p.v_cache) + row * (D / 2) + lane * (E / 2);
    if constexpr (E == 4)
        *reinterpret_cast<uint16_t*>(vq) = uint16_t(q.vpack);
    else
        *vq = uint8_t(q.vpack);
    if (lane % LPG == 0) {
        reinterpret_cast<__half*>(p.v_scale)[meta * NG + lane / LPG] = q.vs;
        reinterpret_cast<__half*>(p.v_zero)[meta * NG + lane / LPG] = q.vz;
    }
}

int grid_for(int64_t work, int per_cta) {
    int64_t g = (work + per_cta - 1) / per_cta;
    if (g < 1) g = 1;
    if (g > 152 * 16) g = 152 * 16;
    return int(g);
}

}  // namespace

cudaError_t launch_reshape_and_cache(const CacheWriteParams& p, int elem_bytes, cudaStream_t stream) {
    const int chunks = p.num_kv_heads * p.head_dim * elem_bytes / 16;
    return launch_kernel(reshape_and_cache_kernel, dim3(grid_for(int64_t(p.num_tokens) * chunks, kThreads)),
                         dim3(kThreads), 0, stream, p, chunks);
}

cudaError_t launch_gather(const GatherParams& p, int elem_bytes, cudaStream_t stream) {
    const int chunks = p.num_kv_heads * p.head_dim * elem_bytes / 16;
    dim3 grid(p.max_blocks, p.num_seqs);
    return launch_kernel(gather_kernel, grid, dim3(kThreads), 0, stream, p, chunks);
}

cudaError_t launch_gather_dequant(const GatherParams& p, cudaStream_t stream) {
    dim3 grid(p.max_blocks, p.num_seqs);
    const bool bf = p.out_dtype == PKV_BF16;
    auto* k = p.head_dim == 128 ? (bf ? gather_dequant_kernel<__nv_bfloat16, 128> : gather_dequant_kernel<__half, 128>)
                                : (bf ? gather_dequant_kernel<__nv_bfloat16, 64> : gather_dequant_kernel<__half, 64>);
    return launch_kernel(k, grid, dim3(kThreads), 0, stream, p);
}

cudaError_t launch_quantize_kv(const CacheWriteParams& p, cudaStream_t stream) {
    const int64_t warps = int64_t(p.num_tokens) * p.num_kv_heads;
    const int64_t g64 = (warps * 32 + kThreads - 1) / kThreads;
    if (g64 > 0x7fffffff) return cudaErrorInvalidValue;
    const int grid = int(g64 < 1 ? 1 : g64);
    const bool bf = p.src_dtype == PKV_BF16;
    auto* k = p.head_dim == 128 ? (bf ? quantize_kernel<__nv_bfloat16, 128> : quantize_kernel<__half, 128>)
                                : (bf ? quantize_kernel<__nv_bfloat16, 64> : quantize_kernel<__half, 64>);
    return launch_kernel(k, dim3(grid), dim3(kThreads), 0, stream, p);
}

}  // namespace pkv
