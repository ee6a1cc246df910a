// decode_cc.cu -- paged decode attention for fp16 / bf16 caches, one query
// token per sequence, on CUDA cores.
//
// What it computes [metalworking "The KV Cache": the pagedattention kernel,
// GQA as a stride trick kv_head = q_head / gqa_factor, split-KV decode; MTPLX
// "How MTPLX Manages Memory Using Request-Sized Paged KV Cache", §"Kernel
// Interface and Memory Slicing": only the stored tokens are read]:
//   out[s, h] = sum_t softmax_t(scale * q[s,h] . K[t, h/g]) V[t, h/g]
// over the tokens [p*P, (p+1)*P) of partition p (whole context when unsplit).
//
// Shape of the kernel (sm_103a):
//   * grid (partition, kv head, sequence); one CTA serves all g query heads of
//     its kv head, so every K/V block is read from HBM exactly once per step.
//   * warp NCW is the producer: it reads the block table 32 entries at a time
//     and issues two 2-D TMA loads per 16-token block (the K tile and the V
//     tile, 16 rows x head_dim, at x = kv_head*head_dim, y = block*16) into an
//     S-stage shared-memory ring guarded by full/empty mbarriers.
//   * warps 0..NCW-1 consume blocks round-robin, each keeping its own online
//     softmax state (running max m, sum l, fp32 accumulator) in registers:
//       QK: LPT lanes per token, each lane a 16-byte chunk (conflict-free),
//           q held in registers pre-scaled by scale*log2(e), xor-shuffle sums;
//       softmax: the block's 16 x g scores in shared memory, one or more per
//           lane, max/sum by xor shuffles over lanes of the same head, exp2;
//       PV: each lane owns head_dim/32 dims of every head, p read as a
//           broadcast, V row read as one 8- or 4-byte word per lane.
//   * at the end the warps' (m, l, acc) are merged in shared memory and the
//     CTA writes either the final row (cast to the output dtype) or the
//     partition's (o_p, m_p, l_p) for the log-sum-exp reduce.
// Every mbarrier wait is bounded; a wait that gives up flags
// PKV_DEVERR_TIMEOUT and the block is skipped.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kBS = 16;

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int D, int G, int NCW>
struct CC {
    static constexpr int CH = D / 8;                             // 16-byte chunks per row
    static constexpr int LPT = (G * D / 64 > 8) ? G * D / 64 : 8;  // lanes per token (QK)
    static constexpr int TPP = 32 / LPT;                         // tokens per pass
    static constexpr int NPASS = kBS / TPP;
    static constexpr int CPL = CH / LPT;                         // chunks per lane
    static constexpr int DPL = D / 32;                           // dims per lane (PV)
    static constexpr int TILE = kBS * D * 2;                     // bytes of a K or V tile
    static constexpr int STAGE = 2 * TILE;
    static constexpr int S = 65536 / STAGE;                      // ring depth
    static constexpr int OFF_BAR = S * STAGE;
    static constexpr int OFF_POISON = OFF_BAR + 2 * S * 8;
    static constexpr int OFF_SC = align_up(OFF_POISON + S * 4, 16);
    static constexpr int OFF_PC = OFF_SC + NCW * kBS * G * 4;          // (p, p) pairs
    static constexpr int OFF_ALPHA = OFF_PC + NCW * kBS * G * 8;
    static constexpr int OFF_MW = OFF_ALPHA + NCW * G * 4;
    static constexpr int OFF_LW = OFF_MW + NCW * G * 4;
    static constexpr int OFF_ACC = align_up(OFF_LW + NCW * G * 4, 16);
    static constexpr int SMEM = OFF_ACC + NCW * G * D * 4;
    static constexpr int THREADS = (NCW + 1) * 32;
    static_assert(CPL >= 1 && CH % LPT == 0, "bad lane split");
    static_assert(TILE % 128 == 0, "tiles must keep 128-byte alignment");
};

template <int N>
__device__ __forceinline__ void load_p(const float* src, float (&p)[N]) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            const float4 v = *reinterpret_cast<const float4*>(src + i);
            p[i] = v.x; p[i + 1] = v.y; p[i + 2] = v.z; p[i + 3] = v.w;
        }
    } else if constexpr (N == 2) {
        const float2 v = *reinterpret_cast<const float2*>(src);
        p[0] = v.x; p[1] = v.y;
    } else {
        p[0] = src[0];
    }
}

template <int N>
__device__ __forceinline__ void load_p2(const float2* src, float2 (&p)[N]) {
    if constexpr (N >= 2) {
#pragma unroll
        for (int i = 0; i < N; i += 2) {
            const float4 v = *reinterpret_cast<const float4*>(src + i);
            p[i] = make_float2(v.x, v.y);
            p[i + 1] = make_float2(v.z, v.w);
        }
    } else {
        p[0] = src[0];
    }
}

template <typename T, int D, int G, int NCW>
__global__ void __launch_bounds__(CC<D, G, NCW>::THREADS)
decode_cc_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                 const AttnParams p) {
    using C = CC<D, G, NCW>;
    constexpr int S = C::S;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* empty = full + S;
    int* poison = reinterpret_cast<int*>(smem + C::OFF_POISON);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int part = blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
    const bool split = p.tmp_out != nullptr;

    int ctx = p.context_lens[s];
    const int cap = p.max_blocks * kBS;
    if (ctx > cap) {
        if (part == 0 && threadIdx.x == 0) flag_error(p.err, PKV_DEVERR_CAPACITY);
        ctx = cap;
    }
    if (ctx < 0) ctx = 0;
    if (split && part == 0 && threadIdx.x == 0 && ctx > p.max_partitions * p.partition_blocks * kBS)
        flag_error(p.err, PKV_DEVERR_CAPACITY);
    const int nblk_seq = (ctx + kBS - 1) / kBS;
    const int b0 = part * p.partition_blocks;
    const int nblk = min(b0 + p.partition_blocks, nblk_seq) - b0;
    const int r = s;  // one query row per sequence
    const int H = p.num_heads;

    if (nblk <= 0) {  // nothing visible in this partition
        if (!split && part == 0)
            for (int i = threadIdx.x; i < G * D; i += C::THREADS)
                store_out(p.out, p.out_dtype, (size_t(r) * H + kvh * G) * D + i, 0.f);
        return;
    }

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == NCW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&k_map);
            prefetch_tensormap(&v_map);
        }
        const int32_t* bt = p.block_tables + size_t(s) * p.max_blocks + b0;
        for (int j0 = 0; j0 < nblk; j0 += 32) {
            const int pbl = (j0 + lane < nblk) ? bt[j0 + lane] : 0;
            const int n = min(32, nblk - j0);
            for (int jj = 0; jj < n; ++jj) {
                int pb = __shfl_sync(0xffffffffu, pbl, jj);
                if (lane == 0) {
                    const int j = j0 + jj, st = j % S;
                    if (j >= S && !mbar_wait(&empty[st], ((j / S) - 1) & 1)) flag_error(p.err, PKV_DEVERR_TIMEOUT);
                    const int bad = (pb < 0 || pb >= p.num_blocks);
                    if (bad) {
                        flag_error(p.err, PKV_DEVERR_OOB_BLOCK);
                        pb = 0;  // load a valid block; the consumer skips it
                    }
                    poison[st] = bad;
                    uint8_t* dst = smem + st * C::STAGE;
                    mbar_arrive_expect_tx(&full[st], C::STAGE);
                    // maps are byte-addressed: x = byte offset of this kv head in a token row
                    tma_load_2d(dst, &k_map, kvh * D * 2, pb * kBS, &full[st]);
                    tma_load_2d(dst + C::TILE, &v_map, kvh * D * 2, pb * kBS, &full[st]);
                }
                __syncwarp();
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int grp = lane / C::LPT, jl = lane % C::LPT;
    // q in registers as (even, odd) dim pairs, pre-scaled by scale*log2(e)
    float2 q2[G][C::CPL * 4];
    {
        const T* qrow = reinterpret_cast<const T*>(p.q) + (size_t(r) * H + kvh * G) * D;
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int k = 0; k < C::CPL; ++k) {
                const uint4 raw = *reinterpret_cast<const uint4*>(qrow + h * D + (jl + k * C::LPT) * 8);
                const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = Half16<T>::unpack2(wds[i]);
                    q2[h][k * 4 + i] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
                }
            }
    }
    // the head whose score this lane holds after the reduce-scatter of the QK sums
    int my_head = 0;
#pragma unroll
    for (int o = C::LPT / 2, nv = G; nv > 1; o >>= 1, nv >>= 1)
        if (jl & o) my_head += nv / 2;
    const bool writer = (jl & (C::LPT / G - 1)) == 0;

    float m_run = -INFINITY, l_run = 0.f;  // for head lane % G
    float2 acc[G][C::DPL / 2];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < C::DPL / 2; ++e) acc[h][e] = make_float2(0.f, 0.f);
    float* sc = reinterpret_cast<float*>(smem + C::OFF_SC) + warp * kBS * G;
    float2* pc = reinterpret_cast<float2*>(smem + C::OFF_PC) + warp * kBS * G;
    float* alph = reinterpret_cast<float*>(smem + C::OFF_ALPHA) + warp * G;

    for (int j = warp; j < nblk; j += NCW) {
        const int st = j % S;
        const bool ok = mbar_wait(&full[st], (j / S) & 1);
        if (!ok && lane == 0) flag_error(p.err, PKV_DEVERR_TIMEOUT);
        const int gb = b0 + j;
        int ntok = (gb == nblk_seq - 1) ? ctx - gb * kBS : kBS;
        if (!ok || poison[st]) ntok = 0;
        if (ntok > 0) {
            const T* Ks = reinterpret_cast<const T*>(smem + st * C::STAGE);
            const T* Vs = Ks + kBS * D;
            // ---- scores: sc[t*G + h] = log2e * scale * q_h . k_t
#pragma unroll
            for (int pass = 0; pass < C::NPASS; ++pass) {
                const int t = pass * C::TPP + grp;
                float2 a2[G];
#pragma unroll
                for (int h = 0; h < G; ++h) a2[h] = make_float2(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < C::CPL; ++k) {
                    const uint4 raw = *reinterpret_cast<const uint4*>(Ks + t * D + (jl + k * C::LPT) * 8);
                    const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 f = Half16<T>::unpack2(wds[i]);
#pragma unroll
                        for (int h = 0; h < G; ++h) a2[h] = __ffma2_rn(q2[h][k * 4 + i], f, a2[h]);
                    }
                }
                float a[G];
#pragma unroll
                for (int h = 0; h < G; ++h) a[h] = a2[h].x + a2[h].y;
                // reduce-scatter over the LPT lanes of the token: halve the live heads per level
#pragma unroll
                for (int o = C::LPT / 2, nv = G; o >= 1; o >>= 1) {
                    const bool up = (jl & o) != 0;
                    if (nv > 1) {
#pragma unroll
                        for (int i = 0; i < nv / 2; ++i) {
                            const float send = up ? a[i] : a[i + nv / 2];
                            const float keep = up ? a[i + nv / 2] : a[i];
                            a[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                        }
                        nv >>= 1;
                    } else {
                        a[0] += __shfl_xor_sync(0xffffffffu, a[0], o);
                    }
                }
                if (writer) sc[t * G + my_head] = (t < ntok) ? a[0] : -INFINITY;
            }
            __syncwarp();
            // ---- online softmax over the block's 16 x G scores
            constexpr int NE = kBS * G;
            constexpr int EPL = (NE + 31) / 32;
            float x[EPL];
            float bm = -INFINITY;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = lane + 32 * i;
                x[i] = (e < NE) ? sc[e] : -INFINITY;
                bm = fmaxf(bm, x[i]);
            }
#pragma unroll
            for (int o = G; o < 32; o <<= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
            const float m_new = fmaxf(m_run, bm);
            float bsum = 0.f;
#pragma unroll
            for (int i = 0; i < EPL; ++i) {
                const int e = lane + 32 * i;
                const float pe = exp2f(x[i] - m_new);
                bsum += pe;
                if (e < NE) pc[e] = make_float2(pe, pe);
            }
#pragma unroll
            for (int o = G; o < 32; o <<= 1) bsum += __shfl_xor_sync(0xffffffffu, bsum, o);
            const float al = exp2f(m_run - m_new);
            l_run = l_run * al + bsum;
            m_run = m_new;
            if (lane < G) alph[lane] = al;
            __syncwarp();
            // ---- acc = acc * alpha + sum_t p_t V_t
            {
                float alv[G];
                load_p<G>(alph, alv);
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < C::DPL / 2; ++e) acc[h][e] = __fmul2_rn(acc[h][e], make_float2(alv[h], alv[h]));
            }
            auto pv_token = [&](int t) {
                float2 vf[C::DPL / 2];
                if constexpr (C::DPL == 4) {
                    const uint2 raw = *reinterpret_cast<const uint2*>(Vs + t * D + lane * 4);
                    vf[0] = Half16<T>::unpack2(raw.x);
                    vf[1] = Half16<T>::unpack2(raw.y);
                } else {
                    vf[0] = Half16<T>::unpack2(*reinterpret_cast<const uint32_t*>(Vs + t * D + lane * 2));
                }
                float2 pp[G];
                load_p2<G>(pc + t * G, pp);
#pragma unroll
                for (int h = 0; h < G; ++h)
#pragma unroll
                    for (int e = 0; e < C::DPL / 2; ++e) acc[h][e] = __ffma2_rn(pp[h], vf[e], acc[h][e]);
            };
            if (ntok == kBS) {
#pragma unroll
                for (int t = 0; t < kBS; ++t) pv_token(t);
            } else {
#pragma unroll 1
                for (int t = 0; t < ntok; ++t) pv_token(t);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }

    // ---------------------------------------------------------------- merge warps
    float* mw = reinterpret_cast<float*>(smem + C::OFF_MW);
    float* lw = reinterpret_cast<float*>(smem + C::OFF_LW);
    float* accw = reinterpret_cast<float*>(smem + C::OFF_ACC);
    if (lane < G) {
        mw[warp * G + lane] = m_run;
        lw[warp * G + lane] = l_run;
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < C::DPL / 2; ++e)
            reinterpret_cast<float2*>(accw + (warp * G + h) * D + lane * C::DPL)[e] = acc[h][e];
    named_barrier_sync(1, NCW * 32);
    for (int idx = threadIdx.x; idx < G * D; idx += NCW * 32) {
        const int h = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w2 = 0; w2 < NCW; ++w2) M = fmaxf(M, mw[w2 * G + h]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w2 = 0; w2 < NCW; ++w2) {
                const float mm = mw[w2 * G + h];
                if (mm != -INFINITY) {
                    const float f = exp2f(mm - M);
                    L = fmaf(lw[w2 * G + h], f, L);
                    O = fmaf(accw[(w2 * G + h) * D + d], f, O);
                }
            }
        }
        const int hg = kvh * G + h;
        const float o = (L > 0.f) ? O / L : 0.f;
        if (split) {
            const size_t pi = (size_t(r) * H + hg) * p.max_partitions + part;
            p.tmp_out[pi * D + d] = o;
            if (d == 0) {
                p.max_logits[pi] = (L > 0.f) ? M * kLn2 : -INFINITY;
                p.exp_sums[pi] = L;
            }
        } else {
            store_out(p.out, p.out_dtype, (size_t(r) * H + hg) * D + d, o);
        }
    }
}

template <typename T, int D, int G>
cudaError_t launch_one(const AttnParams& p, const CUtensorMap& km, const CUtensorMap& vm, int grid_parts,
                       cudaStream_t stream) {
    constexpr int NCW = 4;
    using C = CC<D, G, NCW>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(decode_cc_kernel<T, D, G, NCW>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid(grid_parts, p.num_kv_heads, p.num_seqs);
    decode_cc_kernel<T, D, G, NCW><<<grid, C::THREADS, C::SMEM, stream>>>(km, vm, p);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t dispatch_g(const AttnParams& p, int gqa, const CUtensorMap& km, const CUtensorMap& vm, int gp,
                       cudaStream_t st) {
    switch (gqa) {
        case 1: return launch_one<T, D, 1>(p, km, vm, gp, st);
        case 2: return launch_one<T, D, 2>(p, km, vm, gp, st);
        case 4: return launch_one<T, D, 4>(p, km, vm, gp, st);
        case 8: return launch_one<T, D, 8>(p, km, vm, gp, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool decode_cc_supported(int cache_kind, int head_dim, int gqa) {
    return (cache_kind == PKV_CACHE_F16 || cache_kind == PKV_CACHE_BF16) && (head_dim == 64 || head_dim == 128) &&
           (gqa == 1 || gqa == 2 || gqa == 4 || gqa == 8);
}

cudaError_t launch_decode_cc(const AttnParams& p, int cache_kind, int gqa, const CUtensorMap& k_map,
                             const CUtensorMap& v_map, int grid_parts, cudaStream_t stream) {
    if (cache_kind == PKV_CACHE_BF16) {
        if (p.head_dim == 128) return dispatch_g<__nv_bfloat16, 128>(p, gqa, k_map, v_map, grid_parts, stream);
        return dispatch_g<__nv_bfloat16, 64>(p, gqa, k_map, v_map, grid_parts, stream);
    }
    if (p.head_dim == 128) return dispatch_g<__half, 128>(p, gqa, k_map, v_map, grid_parts, stream);
    return dispatch_g<__half, 64>(p, gqa, k_map, v_map, grid_parts, stream);
}

}  // namespace pkv
