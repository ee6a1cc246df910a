// reduce.cu -- split-KV phase 2: log-sum-exp combination of partition partials;
// also the small set-up kernels that build the work lists of cascade and sparse
// page-indirection attention.
//
// The pages name split-KV decode [mlxcel manual "KV Cache", §"Paged Decode
// Storage and Kernels": decode splits; metalworking "The KV Cache": split-KV
// decode kernels] without printing the combination; this is the exact identity
//   M = max_p m_p,  w_p = l_p exp(m_p - M),  out = sum_p w_p o_p / sum_p w_p
// under which split attention equals single-pass attention.  Partitions with
// l_p = 0 (no visible token for that row) carry no weight.
//
// One CTA of 256 threads per (row, head): the partitions' (m_p, l_p) are read
// in parallel and reduced to M and the weights w_p in shared memory; then
// thread (group k, chunk c) accumulates w_p * o_p over partitions p = k, k+8,
// ... for its 16-byte chunk of head_dim, with four independent loads in
// flight; the eight groups are summed through shared memory.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kThreads = 256;
constexpr int kMaxStaged = 2048;   // partitions whose weights fit the shared buffer at once

template <int D>
__global__ void __launch_bounds__(kThreads) lse_reduce_kernel(ReduceParams p) {
    grid_dep_wait();
    grid_dep_launch();
    constexpr int CH = D / 4;              // float4 chunks of one row
    constexpr int NGRP = kThreads / CH;    // partition groups (8 for D=128, 16 for D=64)
    __shared__ float w_s[kMaxStaged];
    __shared__ float red[kThreads / 32];
    __shared__ float4 part[kThreads];
    const int r = blockIdx.x, h = blockIdx.y;
    const int s = r / p.q_len;
    int ctx = p.context_lens[s];
    if (ctx < 0) ctx = 0;
    int nparts = (ctx + p.partition_size - 1) / p.partition_size;
    if (nparts > p.max_partitions) nparts = p.max_partitions;
    // sliding window: partitions wholly before the last `window` tokens were not written
    const int p_first = (p.window > 0 && ctx > p.window) ? (ctx - p.window) / p.partition_size : 0;
    nparts = nparts > p_first ? nparts - p_first : 0;
    const size_t base = (size_t(r) * p.num_heads + h) * p.max_partitions + p_first;
    // cascade: the row's own partial (slot 0), then its item's (slot 1) if it has one
    if (p.seq_start) nparts = p.seq_start[s] > 0 ? 2 : 1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // M = max over partitions with weight
    float M = -INFINITY;
    for (int i = tid; i < nparts; i += kThreads)
        if (p.exp_sums[base + i] > 0.f) M = fmaxf(M, p.max_logits[base + i]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if (lane == 0) red[warp] = M;
    __syncthreads();
    M = red[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) M = fmaxf(M, red[w]);
    __syncthreads();

    const int grp = tid / CH, c = tid % CH;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float W = 0.f;
    if (M != -INFINITY) {
        for (int p0 = 0; p0 < nparts; p0 += kMaxStaged) {
            const int n = min(kMaxStaged, nparts - p0);
            for (int i = tid; i < n; i += kThreads) {
                const float l = p.exp_sums[base + p0 + i];
                const float w = (l > 0.f) ? l * exp2f((p.max_logits[base + p0 + i] - M) * kLog2e) : 0.f;
                w_s[i] = w;
                W += w;
            }
            __syncthreads();
            int i = grp;
            for (; i + 3 * NGRP < n; i += 4 * NGRP) {   // four independent loads in flight
                float4 v[4];
                float wk[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    wk[u] = w_s[i + u * NGRP];
                    v[u] = *reinterpret_cast<const float4*>(p.tmp_out + (base + p0 + i + u * NGRP) * D + 4 * c);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    if (wk[u] != 0.f) {
                        acc.x = fmaf(wk[u], v[u].x, acc.x);
                        acc.y = fmaf(wk[u], v[u].y, acc.y);
                        acc.z = fmaf(wk[u], v[u].z, acc.z);
                        acc.w = fmaf(wk[u], v[u].w, acc.w);
                    }
            }
            for (; i < n; i += NGRP) {
                const float wk = w_s[i];
                if (wk != 0.f) {
                    const float4 v = *reinterpret_cast<const float4*>(p.tmp_out + (base + p0 + i) * D + 4 * c);
                    acc.x = fmaf(wk, v.x, acc.x);
                    acc.y = fmaf(wk, v.y, acc.y);
                    acc.z = fmaf(wk, v.z, acc.z);
                    acc.w = fmaf(wk, v.w, acc.w);
                }
            }
            __syncthreads();
        }
    }
    // W: block sum of the weights
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
    if (lane == 0) red[warp] = W;
    part[tid] = acc;
    __syncthreads();
    if (tid < CH) {
        float Wt = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) Wt += red[w];
        float4 o = part[tid];
        for (int k = 1; k < NGRP; ++k) {
            const float4 v = part[k * CH + tid];
            o.x += v.x; o.y += v.y; o.z += v.z; o.w += v.w;
        }
        const float inv = (Wt > 0.f) ? 1.f / Wt : 0.f;
        const size_t ob = (size_t(r) * p.num_heads + h) * D + 4 * tid;
        store_out(p.out, p.out_dtype, ob + 0, o.x * inv);
        store_out(p.out, p.out_dtype, ob + 1, o.y * inv);
        store_out(p.out, p.out_dtype, ob + 2, o.z * inv);
        store_out(p.out, p.out_dtype, ob + 3, o.w * inv);
    }
}

}  // namespace

cudaError_t launch_reduce(const ReduceParams& p, cudaStream_t stream) {
    const int rows = p.num_seqs * p.q_len;
    if (p.num_heads > 65535) return cudaErrorInvalidValue;
    dim3 grid(rows, p.num_heads);
    return launch_kernel(p.head_dim == 128 ? lse_reduce_kernel<128> : lse_reduce_kernel<64>, grid, dim3(kThreads), 0,
                         stream, p);
}

namespace {

// Cascade set-up [mlxcel manual "KV Cache", §"Paged Decode Storage and
// Kernels": cascade attention for groups sharing a whole-page prefix], one CTA:
// (1) every sequence gets its list entry (whole context, own table, start 0, one
//     query row); (2) one warp per (item, member) checks that the member's first
//     item_blocks table entries equal the lending (first) member's and that its
//     context covers them, then claims the member for the item.  A member left
//     out keeps start 0 and is attended whole by its own entry, so the result
//     stays exact; the error flag tells the caller its grouping was not what it
//     meant.
constexpr int kSetupThreads = 1024;

// Whether member k of its item shares the item's prefix blocks (one warp).
__device__ __forceinline__ bool cascade_member_ok(const CascadeParams& p, int k, int lane) {
    const int item = k / p.width;
    const int s = p.members[k], s0 = p.members[size_t(item) * p.width], nb = p.item_blocks[item];
    bool ok = s0 >= 0 && s0 < p.num_seqs && nb > 0 && nb <= p.max_blocks && s >= 0 && s < p.num_seqs &&
              p.context_lens[s] >= nb * kBlockSize;
    if (ok) {
        const int32_t* a = p.block_tables + size_t(s) * p.max_blocks;
        const int32_t* b = p.block_tables + size_t(s0) * p.max_blocks;
        bool same = true;
        for (int x = lane; x < nb; x += 32) same &= (a[x] == b[x]);
        ok = __all_sync(0xffffffffu, same);
    }
    return ok;
}

// Its inputs (members, item blocks, block tables, context lengths) are the
// caller's: each warp checks its first member against its item's prefix before
// the grid dependency wait, under the previous kernel's tail; every global
// write comes after it.
__global__ void __launch_bounds__(kSetupThreads) cascade_setup_kernel(CascadeParams p) {
    grid_dep_launch();   // the attention waits for this grid to complete anyway
    const int ni = p.num_items, W = p.width, tid = threadIdx.x;
    const int warp0 = tid >> 5, lane0 = tid & 31;
    const bool ok_first = warp0 < ni * W ? cascade_member_ok(p, warp0, lane0) : false;
    grid_dep_wait();
    for (int i = tid; i < p.num_counters; i += kSetupThreads) p.counters[i] = 0;
    for (int s = tid; s < p.num_seqs; s += kSetupThreads) {
        const int e = ni + s;
        p.list_ctx[e] = p.context_lens[s];
        p.list_seq[e] = s;
        p.list_start[e] = 0;
        p.list_rows[size_t(e) * W] = s;
        for (int j = 1; j < W; ++j) p.list_rows[size_t(e) * W + j] = -1;
    }
    for (int i = tid; i < ni; i += kSetupThreads) {
        const int s0 = p.members[size_t(i) * W], nb = p.item_blocks[i];
        const bool ok = s0 >= 0 && s0 < p.num_seqs && nb >= 0 && nb <= p.max_blocks;
        p.list_ctx[i] = ok ? nb * kBlockSize : 0;
        p.list_seq[i] = ok ? s0 : 0;
        p.list_start[i] = 0;
    }
    __syncthreads();
    const int warp = tid >> 5, lane = tid & 31;
    for (int k = warp; k < ni * W; k += kSetupThreads / 32) {
        const int item = k / W;
        const int s = p.members[k], s0 = p.members[size_t(item) * W], nb = p.item_blocks[item];
        const bool ok = k == warp ? ok_first : cascade_member_ok(p, k, lane);
        int row = -1;
        if (lane == 0) {
            // one item per sequence: the first to claim it
            if (ok && atomicCAS(&p.list_start[ni + s], 0, nb * kBlockSize) == 0) row = s;
            else if (s >= 0 && !(nb == 0 && s0 >= 0 && s0 < p.num_seqs)) flag_error(p.err, PKV_DEVERR_CASCADE);
            p.list_rows[k] = row;
        }
    }
}

// Sparse page-indirection set-up [mlxcel manual "KV Cache", §"Paged Decode
// Storage and Kernels": sparse page-indirection decode], one CTA per sequence,
// 1024 list entries per round.  Entries are taken in order; one outside the
// context's pages or not above the last page taken is skipped (and flagged): an
// in-range entry is kept iff it exceeds every earlier in-range entry (a prefix
// max over the list).  The kept pages' block ids are written back to back, so
// the attention streams a compacted sequence: page k holds compacted tokens
// [16k, 16k + 16), and only the context's tail page can be partial, so the
// compacted context is 16 (n - 1) + (ctx - 16 (pages - 1)) when the tail page
// is kept and 16 n otherwise.
constexpr int kSparseThreads = 1024;
constexpr int kSparseWarps = kSparseThreads / 32;

// Its inputs (lists, counts, block tables, context lengths) are the caller's,
// which no kernel of the library writes: they are read, and the first round's
// kept pages and block ids worked out, before the grid dependency wait, under
// the previous kernel's tail; every global write comes after it.
__global__ void __launch_bounds__(kSparseThreads) sparse_setup_kernel(SparseParams p) {
    grid_dep_launch();   // the attention waits for this grid to complete anyway
    __shared__ int w_max[kSparseWarps], w_cnt[kSparseWarps];
    __shared__ int any_bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, s = blockIdx.x;
    if (tid == 0) any_bad = 0;
    int ctx = p.context_lens[s];
    if (ctx < 0) ctx = 0;
    const bool capped = ctx > p.max_blocks * kBlockSize;
    if (capped) ctx = p.max_blocks * kBlockSize;
    const int npages = (ctx + kBlockSize - 1) / kBlockSize;
    int cnt = p.page_counts[s];
    cnt = cnt < 0 ? 0 : (cnt > p.max_pages ? p.max_pages : cnt);
    const int32_t* list = p.page_lists + size_t(s) * p.max_pages;
    const int32_t* bt = p.block_tables + size_t(s) * p.max_blocks;
    int32_t* out = p.table_out + size_t(s) * p.max_pages;
    int last = -1, n = 0;   // the largest page taken so far, pages taken so far
    for (int base = 0; base < cnt; base += kSparseThreads) {
        const int i = base + tid;
        const int pg = i < cnt ? list[i] : -1;
        const bool in_range = i < cnt && pg >= 0 && pg < npages;
        const int32_t blk = in_range ? bt[pg] : 0;   // an input: fetched ahead of the wait
        // inclusive prefix max of in-range pages within the warp
        int incl = in_range ? pg : -1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl = max(incl, t);
        }
        if (lane == 31) w_max[warp] = incl;
        __syncthreads();
        int before = __shfl_up_sync(0xffffffffu, incl, 1);
        if (lane == 0) before = -1;
        before = max(before, last);
        for (int w2 = 0; w2 < warp; ++w2) before = max(before, w_max[w2]);
        const bool keep = in_range && pg > before;
        if (i < cnt && !keep) any_bad = 1;
        const unsigned m = __ballot_sync(0xffffffffu, keep);
        if (lane == 0) w_cnt[warp] = __popc(m);
        __syncthreads();
        int pos = n + __popc(m & ((1u << lane) - 1u));
        for (int w2 = 0; w2 < warp; ++w2) pos += w_cnt[w2];
        if (base == 0) {   // the first global write: the previous kernel must be done
            grid_dep_wait();
            for (int c = s * kSparseThreads + tid; c < p.num_counters; c += gridDim.x * kSparseThreads)
                p.counters[c] = 0;
        }
        if (keep) out[pos] = blk;
        for (int w2 = 0; w2 < kSparseWarps; ++w2) {
            n += w_cnt[w2];
            last = max(last, w_max[w2]);
        }
        __syncthreads();   // w_max / w_cnt are rewritten by the next round
    }
    if (cnt == 0) {   // no round ran
        grid_dep_wait();
        for (int c = s * kSparseThreads + tid; c < p.num_counters; c += gridDim.x * kSparseThreads) p.counters[c] = 0;
    }
    if (tid == 0) {
        if (capped) flag_error(p.err, PKV_DEVERR_CAPACITY);
        if (any_bad) flag_error(p.err, PKV_DEVERR_PAGE_LIST);
        p.ctx_out[s] = n == 0 ? 0
                              : (last == npages - 1 ? kBlockSize * (n - 1) + (ctx - kBlockSize * (npages - 1))
                                                    : kBlockSize * n);
    }
}

}  // namespace

cudaError_t launch_sparse_setup(const SparseParams& p, cudaStream_t stream) {
    if (p.num_seqs < 1) return cudaSuccess;
    return launch_kernel(sparse_setup_kernel, dim3(p.num_seqs), dim3(kSparseThreads), 0, stream, p);
}

cudaError_t launch_cascade_setup(const CascadeParams& p, cudaStream_t stream) {
    return launch_kernel(cascade_setup_kernel, dim3(1), dim3(kSetupThreads), 0, stream, p);
}

}  // namespace pkv
