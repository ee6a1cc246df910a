// attention_impl.cuh -- the persistent paged-attention kernel and its block
// math, included by attention.cu (attention only), attention_fused.cu (the
// decode step that also writes the cache) and attention_cascade.cu (the
// cascade pass); the instantiations are compiled side by side.  Short page
// names in citations ([MTPLX-2], [MLXCEL], ...) are listed at the top of pkv.h.
//
// What it computes [metalworking "The KV Cache": the pagedattention kernel,
// GQA as the stride trick kv_head = q_head / gqa_factor, split-KV decode;
// MTPLX "How MTPLX Manages Memory Using Request-Sized Paged KV Cache",
// §"Kernel Interface and Memory Slicing": only the stored tokens are read, and
// §"Sliding-Window Memory Control": optionally only the last W of them;
// mlxcel manual "KV Cache", §"Speculative Rewind": a verify block of q_len
// drafts, draft j seeing the history and drafts 0..j]:
//   out[r, h] = sum_t softmax_t(scale * q[r,h] . K[t, h/g]) V[t, h/g]
//
// Work list.  Single pass: CTA c takes a contiguous range of the batch's
// (sequence, kv head) pairs and writes final outputs.  Split and balanced: the
// grid is Hkv lanes of L CTAs; CTA c serves kv head c % Hkv over one range of
// the lane's unit list, laid out sequence by sequence (so the Hkv CTAs of one
// range read the head slices of the same blocks side by side):
//   split        unit = one partition of partition_size tokens ->
//                normalised partial (o_p, m_p, l_p) for the LSE reduce;
//   balanced     unit = one 16-token block; the list's cost (1 per block, plus
//                a fixed charge per extra segment) is cut into equal ranges; a
//                pair cut between CTAs leaves one unnormalised partial per piece
//                in the workspace, and the CTA that finishes its pair's last
//                piece (an atomic count, no waiting) combines them.
//
// CTA anatomy: one CTA per SM, NCW consumer warps + one producer warp.  The
// producer issues up to 16 blocks per pass, one per lane: each lane reads its
// block-table entry, waits for its ring stage and issues the TMA tile loads
// (K8/V4 scales and zeros by cp.async on the same barrier).  Consumer warp w
// takes the blocks of the stages it owns (every NCW-th), with its own online
// softmax state, and the warps merge through shared memory at the end of every
// segment while the producer already streams the next one.
//
// Block math:
//   CcMath  fp16/bf16 decode at group size 1 or 2, CUDA cores: fp32 q pairs,
//           packed fma.rn.f32x2, reduce-scatter shuffles, softmax over 16 x g
//           scores in shared memory;
//   TtMath  fp16/bf16 when a kv head serves 4 to 8 query rows (decode at
//           group size 4 and 8, verify blocks of up to 8 rows): mma.sync
//           m16n8k16 with the contraction turned around (S^T = K Q^T,
//           O^T = V^T P^T), 128B-swizzled tiles via ldmatrix;
//   TcMath  fp16/bf16 for 9 to 16 query rows (the wider verify blocks):
//           mma.sync m16n8k16 on 16 query rows (g heads x q_len drafts);
//   TqMath  K8/V4, any q_len: the contraction turned around (S^T = K Q^T,
//           O^T = V^T P^T) so the query columns sit on the MMA's N side; codes
//           become exact fp16 integers in registers.
// Every mbarrier wait is bounded; a wait that gives up flags
// PKV_DEVERR_TIMEOUT and the block is skipped.
#pragma once

#include "pkv_device.cuh"
#include "pkv_quant.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kBS = 16;
constexpr int kMaxRows = 16;                  // query rows per (sequence, kv head)
constexpr int kSmemLimit = 227 * 1024;
constexpr int kCheckBytes = 16 * 8 + 16 * 4;   // fused step: a warp's slot / block-table checks

// Fused step: a warp's merge buffer (M x D floats) holds the staged new rows
// (q_len x 4D bytes); whether the checks fit behind them too.
__host__ __device__ constexpr bool checks_fit(int M, int QL, int D) { return M * D * 4 >= QL * 4 * D + kCheckBytes; }

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

// Element (m, d) of a per-warp merge buffer [M][D] (floats): 32-byte units of a
// row are XOR-permuted by the row, so the 8 rows a warp's fragment store
// touches at once fall in different banks; 16-byte groups stay together.
__host__ __device__ constexpr int ob_idx(int m, int d, int D) { return m * D + (d ^ ((m & 7) << 3)); }

// ---------------------------------------------------------------- small device helpers

// CASC: the kernel runs cascade attention's pass over its list (the items'
// shared prefixes, then every sequence from its seq_start on), where entry s
// reads the table of item_seq[s] for the query rows row_map[s * q_len + j];
// the other kernels compile without those reads.

// First visible token of list entry s: a sliding window keeps the last `window`
// stored tokens [MTPLX-2 §"Sliding-Window Memory Control"]; a cascade entry
// starts at its seq_start (past its item's shared prefix).
template <bool CASC>
__device__ __forceinline__ int visible_lo(const AttnParams& p, int s, int ctx) {
    if constexpr (CASC) return min(max(p.seq_start[s], 0), ctx);
    return (p.window > 0 && ctx > p.window) ? ctx - p.window : 0;
}

// q / output row of row j of list entry s; < 0: no row
template <bool CASC>
__device__ __forceinline__ int query_row(const AttnParams& p, int s, int j) {
    if constexpr (CASC) return p.row_map[s * p.q_len + j];
    return s * p.q_len + j;
}


template <int W>
__device__ __forceinline__ int swz(int c, int t) {   // 16-byte chunk c of row t under the W-byte TMA swizzle
    return c ^ ((t * W >> 7) & (W / 16 - 1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <bool BF>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    if constexpr (BF)
        mma_bf16(d, a, b0, b1);
    else
        mma_f16(d, a, b0, b1);
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

template <bool BF>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (BF) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

// Four int8 codes (code e in byte e) -> two fp16x2 of the exact integers: flip
// the sign bit (c + 128 in 0..255), splice each byte under the fp16 exponent
// of 1024 (0x64xx = 1024 + byte), subtract 1152.
__device__ __forceinline__ void s8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t x = w ^ 0x80808080u;
    const uint32_t a = __byte_perm(x, 0x64646464u, 0x5140);
    const uint32_t b = __byte_perm(x, 0x64646464u, 0x7362);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), bias);
    lo = *reinterpret_cast<uint32_t*>(&ha);
    hi = *reinterpret_cast<uint32_t*>(&hb);
}

// The same four codes kept biased: fp16x2 of the exact integers c + 1152 (two
// byte permutes and no subtraction); the caller takes 1152 * sum(q) off each
// score instead.
__device__ __forceinline__ void s8x4_to_f16x4_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
    const uint32_t x = w ^ 0x80808080u;
    lo = __byte_perm(x, 0x64646464u, 0x5140);
    hi = __byte_perm(x, 0x64646464u, 0x7362);
}

// 2^x by the hardware's approximate exponential with subnormal results
// flushed to zero (a weight below 2^-126 of the row maximum)
__device__ __forceinline__ float exp2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Nibble i of both 16-bit halves of w -> fp16x2 of the exact integers 0..15.
__device__ __forceinline__ uint32_t u4pair_to_f16x2(uint32_t w, int i) {
    const uint32_t x = ((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u;   // 1024 + code
    const __half2 bias = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
    __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&x), bias);
    return *reinterpret_cast<uint32_t*>(&h);
}

template <int N>
__device__ __forceinline__ void load_f(const float* src, float (&v)[N]) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            const float4 x = *reinterpret_cast<const float4*>(src + i);
            v[i] = x.x; v[i + 1] = x.y; v[i + 2] = x.z; v[i + 3] = x.w;
        }
    } else if constexpr (N == 2) {
        const float2 x = *reinterpret_cast<const float2*>(src);
        v[0] = x.x; v[1] = x.y;
    } else {
        v[0] = src[0];
    }
}

template <int N>
__device__ __forceinline__ void load_f2(const float2* src, float2 (&v)[N]) {
    if constexpr (N >= 2) {
#pragma unroll
        for (int i = 0; i < N; i += 2) {
            const float4 x = *reinterpret_cast<const float4*>(src + i);
            v[i] = make_float2(x.x, x.y);
            v[i + 1] = make_float2(x.z, x.w);
        }
    } else {
        v[0] = src[0];
    }
}

// ---------------------------------------------------------------- CUDA-core block math

template <typename T, int D, int G>
struct CcMath {
    static constexpr bool kTensor = false;
    static constexpr int kD = D;
    // 11 consumer warps + the producer: 12 warps, three per SM sub-partition,
    // which leaves 168 registers a thread (this math runs group sizes 1 and 2)
    static constexpr int NCW = 11;
    static constexpr int kSegCost = pkv::kSegCost;   // balanced: blocks' worth one more segment costs
    static constexpr int kIssueGroup = 16;           // blocks the producer issues per pass
    static constexpr int CH = D / 8;                               // 16-byte chunks per row
    static constexpr int LPT = (G * D / 64 > 8) ? G * D / 64 : 8;  // lanes per token (QK)
    static constexpr int TPP = 32 / LPT;                           // tokens per pass
    static constexpr int NPASS = kBS / TPP;
    static constexpr int CPL = CH / LPT;                           // chunks per lane
    static constexpr int DPL = D / 32;                             // dims per lane (PV)
    static constexpr int KT = kBS * D * 2;                         // K (or V) tile bytes
    static constexpr int TX = 2 * KT;                              // bytes landing per stage
    static constexpr int STAGE = 2 * KT;
    static constexpr int SCRATCH = align_up(kBS * G * 4 + kBS * G * 8 + G * 4, 16);   // per warp
    static_assert(CPL >= 1 && CH % LPT == 0, "bad lane split");

    float2 q2[G][CPL * 4];
    float m_run, l_run;            // for head lane % G
    int lo_;                       // first visible token (sliding window)
    float2 acc[G][DPL / 2];
    int my_head;
    bool writer;

    static __device__ __forceinline__ void issue(uint8_t* dst, const CUtensorMap* km, const CUtensorMap* vm,
                                                 const AttnParams&, int kvh, int pb, uint64_t* bar) {
        // byte-addressed maps, box = one kv head's 16 rows
        mbar_arrive_expect_tx(bar, TX);
        const uint64_t pol = l2_evict_first_policy();
        tma_load_2d_hint(dst, km, kvh * D * 2, pb * kBS, bar, pol);
        tma_load_2d_hint(dst + KT, vm, kvh * D * 2, pb * kBS, bar, pol);
    }

    static constexpr bool kQ8 = false;
    // copy staged row j into tile row r of a stage (K rows then V rows, 2D bytes each)
    __device__ __forceinline__ void patch(uint8_t* stg, int r, int j, const uint8_t* buf, int lane,
                                          const AttnParams&) const {
        // explicit shared-space copies: a generic store here costs the block loop
        // its schedule (measured: 2 us on a 25 us launch)
        constexpr int CHK = D * 2 / 16;
        if (lane < 2 * CHK)
            lds_sts_16(smem_addr(stg) + (lane < CHK ? 0 : KT) + r * 2 * D + 16 * (lane % CHK),
                       smem_addr(buf) + j * 4 * D + 16 * lane);
    }

    __device__ __forceinline__ void init(int lane) {
        const int jl = lane % LPT;
        my_head = 0;
#pragma unroll
        for (int o = LPT / 2, nv = G; nv > 1; o >>= 1, nv >>= 1)
            if (jl & o) my_head += nv / 2;
        writer = (jl & (LPT / G - 1)) == 0;
    }

    template <bool CASC>
    __device__ __forceinline__ void begin(const AttnParams& p, int s, int kvh, int ctx, int lane) {
        const int jl = lane % LPT;
        lo_ = visible_lo<CASC>(p, s, ctx);
        const T* qrow = reinterpret_cast<const T*>(p.q) + (size_t(s) * p.num_heads + kvh * G) * D;
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int k = 0; k < CPL; ++k) {
                const uint4 raw = *reinterpret_cast<const uint4*>(qrow + h * D + (jl + k * LPT) * 8);
                const uint32_t wds[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float2 f = Half16<T>::unpack2(wds[i]);
                    q2[h][k * 4 + i] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
                }
            }
        m_run = -INFINITY;
        l_run = 0.f;
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < DPL / 2; ++e) acc[h][e] = make_float2(0.f, 0.f);
    }

    __device__ __forceinline__ void block(const uint8_t* stg, int pos0, int ntok, uint8_t* scratch, int lane) {
        float* sc = reinterpret_cast<float*>(scratch);
        float2* pc = reinterpret_cast<float2*>(scratch + kBS * G * 4);
        float* alph = reinterpret_cast<float*>(scratch + kBS * G * 12);
        const int grp = lane / LPT, jl = lane % LPT;
        const T* Ks = reinterpret_cast<const T*>(stg);
        const T* Vs = Ks + kBS * D;
        // ---- scores: sc[t*G + h] = log2e * scale * q_h . k_t
#pragma unroll
        for (int pass = 0; pass < NPASS; ++pass) {
            const int t = pass * TPP + grp;
            float2 a2[G];
#pragma unroll
            for (int h = 0; h < G; ++h) a2[h] = make_float2(0.f, 0.f);
#pragma unroll
            for (int k = 0; k < CPL; ++k) {
                const uint4 raw = *reinterpret_cast<const uint4*>(Ks + t * D + (jl + k * LPT) * 8);
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
            // reduce-scatter over the token's LPT lanes: halve the live heads per level
#pragma unroll
            for (int o = LPT / 2, nv = G; o >= 1; o >>= 1) {
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
            if (writer) sc[t * G + my_head] = (t < ntok && pos0 + t >= lo_) ? a[0] : -INFINITY;
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
            load_f<G>(alph, alv);
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < DPL / 2; ++e) acc[h][e] = __fmul2_rn(acc[h][e], make_float2(alv[h], alv[h]));
        }
        auto pv_token = [&](int t) {
            float2 vf[DPL / 2];
            if constexpr (DPL == 4) {
                const uint2 raw = *reinterpret_cast<const uint2*>(Vs + t * D + lane * 4);
                vf[0] = Half16<T>::unpack2(raw.x);
                vf[1] = Half16<T>::unpack2(raw.y);
            } else {
                vf[0] = Half16<T>::unpack2(*reinterpret_cast<const uint32_t*>(Vs + t * D + lane * 2));
            }
            float2 pp[G];
            load_f2<G>(pc + t * G, pp);
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < DPL / 2; ++e) acc[h][e] = __ffma2_rn(pp[h], vf[e], acc[h][e]);
        };
        if (ntok == kBS) {
#pragma unroll
            for (int t = 0; t < kBS; ++t) pv_token(t);
        } else {
#pragma unroll 1
            for (int t = 0; t < ntok; ++t) pv_token(t);
        }
        __syncwarp();
    }

    __device__ __forceinline__ void finish(int) {}

    // unnormalised accumulator rows [G][D] and per-row (m, l) of this warp
    __device__ __forceinline__ void store(float* ob, float* mw, float* lw, int /*M*/, int lane) const {
        if (lane < G) {
            mw[lane] = m_run;
            lw[lane] = l_run;
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < DPL / 2; ++e)
                *reinterpret_cast<float2*>(ob + ob_idx(h, lane * DPL + 2 * e, D)) = acc[h][e];
    }
};

// ---------------------------------------------------------------- tensor-core block math

// Multi-token verify blocks on fp16 / bf16 caches: the 16-row query tile (g
// heads x q_len drafts) against a 16-token block.
template <int KIND, int D>
struct TcMath {
    static constexpr bool kTensor = true;
    static constexpr int kD = D;
    // 7 consumer warps + the producer: 8 warps, two per SM sub-partition, so a
    // thread may use up to 255 registers (the MMA fragments need ~230)
    static constexpr int NCW = 7;
    static constexpr int kSegCost = pkv::kSegCost;
    // Blocks the producer issues per pass: a pass waits on every stage it
    // refills, so a smaller pass refills the first of them sooner (8 measured
    // faster than 16 on the 32K and batch-8 decodes)
    static constexpr int kIssueGroup = 8;
    static constexpr bool BF = KIND == PKV_CACHE_BF16;
    static constexpr int NKS = D / 16;
    static constexpr int NNT = D / 8;
    static constexpr int KT = kBS * 2 * D;
    static constexpr int VT = kBS * 2 * D;
    static constexpr int OFF_V = align_up(KT, 1024);
    static constexpr int TX = KT + VT;   // bytes the TMA copies deliver
    static constexpr int STAGE = align_up(OFF_V + VT, 1024);
    static constexpr int SCRATCH = 0;
    static_assert(KIND != PKV_CACHE_K8V4, "K8/V4 runs TqMath");
    static_assert(OFF_V % 1024 == 0 && STAGE % 1024 == 0, "swizzled tiles need 1 KB alignment");

    uint32_t qa[NKS][4];
    float o[NNT][4];
    float m_run[2], l_run[2];
    int lim[2];
    int lo_;   // first visible token (sliding window)

    static __device__ __forceinline__ void issue(uint8_t* dst, const CUtensorMap* km, const CUtensorMap* vm,
                                                 const AttnParams&, int kvh, int pb, uint64_t* bar) {
        // one 3-D box per tile: {128 bytes, 16 rows, D/64 chunks} lands as
        // D/64 consecutive 2 KB sub-tiles of 128-byte rows, 128B swizzle
        mbar_arrive_expect_tx(bar, TX);
        const uint64_t pol = l2_evict_first_policy();
        tma_load_3d_hint(dst, km, 0, pb * kBS, kvh * (D / 64), bar, pol);
        tma_load_3d_hint(dst + OFF_V, vm, 0, pb * kBS, kvh * (D / 64), bar, pol);
    }

    static constexpr bool kQ8 = false;
    // tile row r, 16-byte chunk c (8 dims) sits at (c/8)*2048 + r*128 + 16*((c%8) ^ (r%8))
    __device__ __forceinline__ void patch(uint8_t* stg, int r, int j, const uint8_t* buf, int lane,
                                          const AttnParams&) const {
        constexpr int CHK = D * 2 / 16;
        if (lane < 2 * CHK) {
            const int c = lane % CHK;
            lds_sts_16(smem_addr(stg) + (lane < CHK ? 0 : OFF_V) + (c >> 3) * 2048 + r * 128 + 16 * swz<128>(c & 7, r),
                       smem_addr(buf) + j * 4 * D + 16 * lane);
        }
    }

    __device__ __forceinline__ void init(int) {}

    // rows g and g+8 of the 16-row tile: row m = head (m / q_len), draft (m % q_len)
    template <bool CASC>
    __device__ __forceinline__ void begin(const AttnParams& p, int s, int kvh, int ctx, int lane) {
        const int g = lane >> 2, tid = lane & 3;
        const int G = p.num_heads / p.num_kv_heads, QL = p.q_len, M = G * QL;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int m = g + 8 * r;
            const int h = m < M ? m / QL : 0, j = m < M ? m % QL : 0;
            const int qr = m < M ? query_row<CASC>(p, s, j) : -1;
            const bool valid = qr >= 0;
            // a cascade row (one decode query) sees the entry's whole context; verify rows are causal
            lim[r] = valid ? (CASC ? ctx : max(0, ctx - QL + j + 1)) : 0;
            const size_t qoff = (size_t(valid ? qr : 0) * p.num_heads + kvh * G + h) * D;
            const uint32_t* qw = reinterpret_cast<const uint32_t*>(p.q);
            lo_ = visible_lo<CASC>(p, s, ctx);
#pragma unroll
            for (int kk = 0; kk < NKS; ++kk) {
                qa[kk][r] = valid ? qw[(qoff + 16 * kk + 2 * tid) / 2] : 0u;
                qa[kk][2 + r] = valid ? qw[(qoff + 16 * kk + 8 + 2 * tid) / 2] : 0u;
            }
        }
#pragma unroll
        for (int n = 0; n < NNT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
        m_run[0] = m_run[1] = -INFINITY;
        l_run[0] = l_run[1] = 0.f;
    }

    __device__ __forceinline__ void block(const uint8_t* stg, int pos0, int ntok, uint8_t*, int lane) {
        const int tid = lane & 3;
        const uint32_t stg_a = smem_addr(stg);
        float sc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
        // ------------------------------------------------ S = Q K^T
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int kp = 0; kp < NKS / 2; ++kp) {
                const int mi = lane >> 3, r = lane & 7;
                const int t = nt * 8 + r, c = 4 * kp + mi;           // 8-dim chunk c
                const uint32_t addr = stg_a + (c >> 3) * 2048 + t * 128 + 16 * swz<128>(c & 7, t);
                uint32_t R[4];
                ldsm_x4(addr, R);
                mma16816<BF>(sc[nt], qa[2 * kp], R[0], R[1]);
                mma16816<BF>(sc[nt], qa[2 * kp + 1], R[2], R[3]);
            }
        }
        // ------------------------------------------------ scale, mask, online softmax (rows g, g+8)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int pos = pos0 + nt * 8 + 2 * tid + (e & 1);
                sc[nt][e] = (pos < lim[e >> 1] && pos >= lo_) ? sc[nt][e] * scale_log2_ : -INFINITY;
            }
        float alpha[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            float bm = fmaxf(fmaxf(sc[0][2 * r], sc[0][2 * r + 1]), fmaxf(sc[1][2 * r], sc[1][2 * r + 1]));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
            const float mn = fmaxf(m_run[r], bm);
            const float mu = (mn == -INFINITY) ? 0.f : mn;
            // nothing accumulated yet (padding rows stay so): no rescale
            alpha[r] = (m_run[r] == -INFINITY) ? 1.f : exp2f(m_run[r] - mu);
            float rs = 0.f;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float pe = exp2f(sc[nt][2 * r + e] - mu);
                    sc[nt][2 * r + e] = pe;
                    rs += pe;
                }
            rs += __shfl_xor_sync(0xffffffffu, rs, 1);
            rs += __shfl_xor_sync(0xffffffffu, rs, 2);
            l_run[r] = l_run[r] * alpha[r] + rs;
            m_run[r] = mn;
        }
        if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
            for (int n = 0; n < NNT; ++n) {
                o[n][0] *= alpha[0]; o[n][1] *= alpha[0];
                o[n][2] *= alpha[1]; o[n][3] *= alpha[1];
            }
        }
        // ------------------------------------------------ O += P V
        // P as the A operand: bf16 keeps 8 significant bits, so P = hi + lo
        // (two MMAs, P exact to ~2^-17); fp16's 11 bits are kept as one operand.
        uint32_t a[4], alo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float x = sc[i >> 1][2 * (i & 1)], y = sc[i >> 1][2 * (i & 1) + 1];
            a[i] = pack2<BF>(x, y);
            if constexpr (BF) {
                const float hx = __uint_as_float(a[i] << 16), hy = __uint_as_float(a[i] & 0xffff0000u);
                alo[i] = pack2<BF>(x - hx, y - hy);
            }
        }
        // V rows past the context may hold anything (NaN): zero them in the operand
        const uint32_t m01 = (2 * tid < ntok ? 0x0000ffffu : 0u) | (2 * tid + 1 < ntok ? 0xffff0000u : 0u);
        const uint32_t m23 = (8 + 2 * tid < ntok ? 0x0000ffffu : 0u) | (9 + 2 * tid < ntok ? 0xffff0000u : 0u);
#pragma unroll
        for (int np = 0; np < NNT / 2; ++np) {
            const int mi = lane >> 3, r = lane & 7;
            const int t = (mi & 1) * 8 + r, c = 2 * np + (mi >> 1);   // 8-dim chunk = n-tile
            const uint32_t addr = stg_a + OFF_V + (c >> 3) * 2048 + t * 128 + 16 * swz<128>(c & 7, t);
            uint32_t R[4];
            ldsm_x4_t(addr, R);
            if (ntok < kBS) {
                R[0] &= m01; R[1] &= m23; R[2] &= m01; R[3] &= m23;
            }
            mma16816<BF>(o[2 * np], a, R[0], R[1]);
            mma16816<BF>(o[2 * np + 1], a, R[2], R[3]);
            if constexpr (BF) {
                mma16816<BF>(o[2 * np], alo, R[0], R[1]);
                mma16816<BF>(o[2 * np + 1], alo, R[2], R[3]);
            }
        }
    }

    __device__ __forceinline__ void finish(int) {}

    // unnormalised rows [M][D] (ob_idx order) and per-row (m, l) of this warp
    __device__ __forceinline__ void store(float* ob, float* mw, float* lw, int M, int lane) const {
        const int g = lane >> 2, tid = lane & 3;
#pragma unroll
        for (int n = 0; n < NNT; ++n)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const int m = g + 8 * r;
                if (m < M)
                    *reinterpret_cast<float2*>(ob + ob_idx(m, 8 * n + 2 * tid, D)) =
                        make_float2(o[n][2 * r], o[n][2 * r + 1]);
            }
        if (tid == 0) {
            if (g < M) {
                mw[g] = m_run[0];
                lw[g] = l_run[0];
            }
            if (g + 8 < M) {
                mw[g + 8] = m_run[1];
                lw[g + 8] = l_run[1];
            }
        }
    }

    float scale_log2_;
};

// ---------------------------------------------------------------- K8/V4 block math, transposed

__device__ __forceinline__ uint32_t movm_trans(uint32_t x) {   // 8x8 b16 matrix transpose across the warp
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    __half2 x, y;
    memcpy(&x, &a, 4);
    memcpy(&y, &b, 4);
    const __half2 z = __hmul2(x, y);
    uint32_t r;
    memcpy(&r, &z, 4);
    return r;
}

// fp16 / bf16 cache, up to 8 query rows per kv head (decode at group size 4
// and 8, verify blocks of g * q_len <= 8).  The same tiles as TcMath, with the
// contraction turned around as for K8/V4: S^T = K Q^T puts the block's 16
// tokens on the MMA's M side and the query rows on its 8 columns, and
// O^T = V^T P^T puts 16 head dims on M.  Per 16-token block that is D/16 MMAs
// for the scores and D/16 for the values (twice that for P's low bf16 half),
// where a 16-row query tile spends as many on 12 padding rows.
//   K: the A operand straight from the swizzled tile (ldmatrix).
//   V: the A operand V^T from the tile (ldmatrix.trans); rows past the
//      context are zeroed in the operand (they may hold NaN).
//   P: the S^T accumulator is packed and turned into the P^T operand with
//      movmatrix; bf16 keeps 8 significant bits, so P = hi + lo (two MMAs, P
//      exact to ~2^-17), fp16's 11 bits are kept as one operand.
template <int KIND, int D>
struct TtMath {
    static constexpr bool kTensor = true;
    static constexpr int kD = D;
    static constexpr int NCW = 7;
    static constexpr int kSegCost = pkv::kSegCost;
    static constexpr int kIssueGroup = 8;
    static constexpr bool BF = KIND == PKV_CACHE_BF16;
    static constexpr int NKS = D / 16;     // k-steps of the score contraction
    static constexpr int NMT = D / 16;     // M tiles of O^T
    static constexpr int KT = kBS * 2 * D;
    static constexpr int VT = kBS * 2 * D;
    static constexpr int OFF_V = align_up(KT, 1024);
    static constexpr int TX = KT + VT;   // bytes the TMA copies deliver
    static constexpr int STAGE = align_up(OFF_V + VT, 1024);
    static constexpr int SCRATCH = 0;
    static_assert(KIND != PKV_CACHE_K8V4, "K8/V4 runs TqMath");
    static_assert(OFF_V % 1024 == 0 && STAGE % 1024 == 0, "swizzled tiles need 1 KB alignment");

    uint32_t qb[NKS][2];   // Q^T operand: query column g, this thread's dims
    float o[NMT][4];       // O^T: dims (g, g + 8) of each M tile x query columns (2t, 2t + 1)
    float m_run[2], l_part[2];   // query columns 2t, 2t + 1 (l: this thread's tokens)
    int lim[2];
    int lo_;   // first visible token (sliding window)
    float scale_log2_;

    static __device__ __forceinline__ void issue(uint8_t* dst, const CUtensorMap* km, const CUtensorMap* vm,
                                                 const AttnParams& p, int kvh, int pb, uint64_t* bar) {
        TcMath<KIND, D>::issue(dst, km, vm, p, kvh, pb, bar);
    }

    static constexpr bool kQ8 = false;
    __device__ __forceinline__ void patch(uint8_t* stg, int r, int j, const uint8_t* buf, int lane,
                                          const AttnParams& p) const {
        constexpr int CHK = D * 2 / 16;
        if (lane < 2 * CHK) {
            const int c = lane % CHK;
            lds_sts_16(smem_addr(stg) + (lane < CHK ? 0 : OFF_V) + (c >> 3) * 2048 + r * 128 + 16 * swz<128>(c & 7, r),
                       smem_addr(buf) + j * 4 * D + 16 * lane);
        }
    }

    __device__ __forceinline__ void init(int) {}

    // query column n = row m of the pair (head m / q_len, draft m % q_len)
    template <bool CASC>
    __device__ __forceinline__ void begin(const AttnParams& p, int s, int kvh, int ctx, int lane) {
        const int g = lane >> 2, t = lane & 3;
        const int G = p.num_heads / p.num_kv_heads, QL = p.q_len, M = G * QL;
        lo_ = visible_lo<CASC>(p, s, ctx);
        {
            // this thread's B fragments: column g
            const int h = g < M ? g / QL : 0, j = g < M ? g % QL : 0;
            const int qr = g < M ? query_row<CASC>(p, s, j) : -1;
            const bool valid = qr >= 0;
            const size_t qoff = (size_t(valid ? qr : 0) * p.num_heads + kvh * G + h) * D;
            const uint32_t* qw = reinterpret_cast<const uint32_t*>(p.q);
#pragma unroll
            for (int kk = 0; kk < NKS; ++kk) {
                qb[kk][0] = valid ? qw[(qoff + 16 * kk + 2 * t) / 2] : 0u;
                qb[kk][1] = valid ? qw[(qoff + 16 * kk + 8 + 2 * t) / 2] : 0u;
            }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            // this thread's accumulator columns 2t + e
            const int n = 2 * t + e;
            const int j = n < M ? n % QL : 0;
            const bool ok = n < M && query_row<CASC>(p, s, j) >= 0;
            // a cascade row (one decode query) sees the entry's whole context; verify rows are causal
            lim[e] = ok ? (CASC ? ctx : max(0, ctx - QL + j + 1)) : 0;
            m_run[e] = -INFINITY;
            l_part[e] = 0.f;
        }
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    }

    __device__ __forceinline__ void block(const uint8_t* stg, int pos0, int ntok, uint8_t*, int lane) {
        const int g = lane >> 2, t = lane & 3;
        const int mi = lane >> 3, r = lane & 7;
        const uint32_t stg_a = smem_addr(stg);
        // ------------------------------------------------ S^T = K Q^T (rows = tokens g, g + 8)
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < NKS; ++kk) {
            // matrices: tokens 0-7 / 8-15 of 8-dim chunk 2kk, then of chunk 2kk + 1
            const int tk = (mi & 1) * 8 + r, c = 2 * kk + (mi >> 1);
            uint32_t a[4];
            ldsm_x4(stg_a + (c >> 3) * 2048 + tk * 128 + 16 * swz<128>(c & 7, tk), a);
            mma16816<BF>(sc, a, qb[kk][0], qb[kk][1]);
        }
        // scale, context / causal / window mask
        const int pg = pos0 + g, pg8 = pos0 + g + 8;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            sc[e] = (pg < lim[e] && pg >= lo_) ? sc[e] * scale_log2_ : -INFINITY;
            sc[2 + e] = (pg8 < lim[e] && pg8 >= lo_) ? sc[2 + e] * scale_log2_ : -INFINITY;
        }
        // ------------------------------------------------ online softmax per query column
        float alpha[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float bm = fmaxf(sc[e], sc[2 + e]);
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
            bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
            const float mn = fmaxf(m_run[e], bm);
            const float mu = (mn == -INFINITY) ? 0.f : mn;
            // nothing accumulated yet (padding columns stay so): no rescale
            alpha[e] = (m_run[e] == -INFINITY) ? 1.f : exp2f(m_run[e] - mu);
            const float p0 = exp2f(sc[e] - mu), p1 = exp2f(sc[2 + e] - mu);
            sc[e] = p0;
            sc[2 + e] = p1;
            l_part[e] = l_part[e] * alpha[e] + (p0 + p1);
            m_run[e] = mn;
        }
        if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
            for (int mt = 0; mt < NMT; ++mt) {
                o[mt][0] *= alpha[0]; o[mt][2] *= alpha[0];
                o[mt][1] *= alpha[1]; o[mt][3] *= alpha[1];
            }
        }
        // ------------------------------------------------ P^T operand (tokens 2t.., query column g)
        const uint32_t p01 = pack2<BF>(sc[0], sc[1]), p23 = pack2<BF>(sc[2], sc[3]);
        const uint32_t b0 = movm_trans(p01), b1 = movm_trans(p23);
        uint32_t c0 = 0u, c1 = 0u;
        if constexpr (BF) {
            const uint32_t l01 = pack2<BF>(sc[0] - __uint_as_float(p01 << 16), sc[1] - __uint_as_float(p01 & 0xffff0000u));
            const uint32_t l23 = pack2<BF>(sc[2] - __uint_as_float(p23 << 16), sc[3] - __uint_as_float(p23 & 0xffff0000u));
            c0 = movm_trans(l01);
            c1 = movm_trans(l23);
        }
        // V rows past the context may hold anything (NaN): zero them in the operand
        const uint32_t m01 = (2 * t < ntok ? 0x0000ffffu : 0u) | (2 * t + 1 < ntok ? 0xffff0000u : 0u);
        const uint32_t m23 = (8 + 2 * t < ntok ? 0x0000ffffu : 0u) | (9 + 2 * t < ntok ? 0xffff0000u : 0u);
        // ------------------------------------------------ O^T += V^T P^T
#pragma unroll
        for (int mt = 0; mt < NMT; ++mt) {
            // matrices (transposed): tokens 0-7 of chunks 2mt, 2mt + 1, then tokens 8-15
            const int tk = (mi >> 1) * 8 + r, c = 2 * mt + (mi & 1);
            uint32_t a[4];
            ldsm_x4_t(stg_a + OFF_V + (c >> 3) * 2048 + tk * 128 + 16 * swz<128>(c & 7, tk), a);
            if (ntok < kBS) {
                a[0] &= m01; a[1] &= m01; a[2] &= m23; a[3] &= m23;
            }
            mma16816<BF>(o[mt], a, b0, b1);
            if constexpr (BF) mma16816<BF>(o[mt], a, c0, c1);
        }
    }

    __device__ __forceinline__ void finish(int) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            float l = l_part[e];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            l_part[e] = l;
        }
    }

    // unnormalised rows [M][D] (ob_idx order) and per-row (m, l) of this warp
    __device__ __forceinline__ void store(float* ob, float* mw, float* lw, int M, int lane) const {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int q = 2 * t + e;
            if (q >= M) continue;
#pragma unroll
            for (int mt = 0; mt < NMT; ++mt) {
                ob[ob_idx(q, 16 * mt + g, D)] = o[mt][e];
                ob[ob_idx(q, 16 * mt + g + 8, D)] = o[mt][2 + e];
            }
            if (g == 0) {
                mw[q] = m_run[e];
                lw[q] = l_part[e];
            }
        }
    }
};

// K8/V4 cache (see quantize_kernel).  The query tile of a decode block is only
// g*q_len rows, so the contraction is turned around: S^T = K Q^T puts the 16
// tokens on the MMA's M side and up to 8 (NT = 1) or 16 (NT = 2) query columns
// on N, and O^T = V^T P^T puts 16 head dims on M.  Per 16-token block and 8
// query columns that is D/16 MMAs for the scores and D/16 for the values,
// where a 16-row query tile needs twice as many.
//   K: int8 codes -> exact fp16 integers; the per-token K scale multiplies the
//      scores.  A thread's four k positions of a k-step are four consecutive
//      bytes of a row; the query operand uses the same dim order.
//   V: 4-bit codes -> exact fp16 integers in the A operand (ldmatrix.trans of
//      16-bit words = 4 dims x 2 tokens).  A 16-byte chunk of a V row is one
//      32-dim group, and an M tile takes dims {4w+i, 4w+i+2} of one group, so
//      the per-(token, group) scale goes into the P^T operand (P * s in fp16)
//      and the zero point into one more MMA, Z^T P^T, added at the end.
//   P: the S^T accumulator is packed to fp16 and turned into the P^T operand
//      with movmatrix.
template <int D, int NT>
struct TqMath {
    static constexpr bool kTensor = true;
    static constexpr int kD = D;
    // NT = 1: 11 consumer warps at <= 168 registers; NT = 2: 7 at <= 255
    static constexpr int NCW = NT == 1 ? 11 : 7;
    // The K8/V4 math is bound by its consumers, so a segment switch (merge,
    // piece, the next segment's queries) is not hidden behind the stream: it is
    // charged more (32 measured best of 24, 32, 40, 48)
    static constexpr int kSegCost = 32;
    // 18 metadata copies and two tensor copies per block: 22 blocks per pass,
    // two per consumer warp (8, 11, 12, 16 and 32 measured slower)
    static constexpr int kIssueGroup = 22;
    static constexpr int NG = D / 32;      // V groups
    static constexpr int NKS = D / 16;     // k-steps of the score contraction
    static constexpr int KT = kBS * D;
    static constexpr int VT = kBS * D / 2;
    static constexpr int KS = kBS * 2;
    static constexpr int VS = kBS * NG * 2;
    static constexpr int OFF_V = align_up(KT, 1024);
    static constexpr int OFF_KS = OFF_V + align_up(VT, 16);
    static constexpr int OFF_VS = OFF_KS + KS;
    static constexpr int OFF_VZ = OFF_VS + VS;
    static constexpr int TX = KT + VT;   // bytes the TMA copies deliver
    static constexpr int STAGE = align_up(OFF_VZ + VS, 1024);
    static constexpr int SCRATCH = 0;
    static_assert(OFF_V % 1024 == 0 && STAGE % 1024 == 0, "swizzled tiles need 1 KB alignment");
    static_assert(OFF_VS % 16 == 0 && OFF_VZ % 16 == 0, "scale rows are read 16 bytes at a time");

    uint32_t qb[NT][NKS][2];   // Q^T operand: query column g (+8), this thread's dims
    float o[NT][2 * NG][4];    // O^T accumulators: M tile (group, i) x 8 query columns
    float cz[NT][4];           // Z^T P^T: rows = groups
    float m_run[NT][2], l_part[NT][2];   // per query column 2t, 2t+1 (l: this thread's tokens)
    int lim[NT][2];
    float kbias[NT][2];   // 1152 * sum of q over the head dims, query columns 2t, 2t+1
    int lo_;       // first visible token (sliding window)
    int lim_lo_;   // smallest lim over this thread's live columns (no live column: INT_MAX)
    float scale_log2_;

    static __device__ __forceinline__ void issue(uint8_t* dst, const CUtensorMap* km, const CUtensorMap* vm,
                                                 const AttnParams& p, int kvh, int pb, uint64_t* bar) {
        const size_t meta = size_t(pb) * p.num_kv_heads + kvh;
        const uint8_t* ks = reinterpret_cast<const uint8_t*>(p.k_scale) + meta * KS;
        const uint8_t* vs = reinterpret_cast<const uint8_t*>(p.v_scale) + meta * VS;
        const uint8_t* vz = reinterpret_cast<const uint8_t*>(p.v_zero) + meta * VS;
        const uint64_t pol = l2_evict_first_policy();
#pragma unroll
        for (int c = 0; c < KS; c += 16) cp_async_16_hint(dst + OFF_KS + c, ks + c, pol);
#pragma unroll
        for (int c = 0; c < VS; c += 16) {
            cp_async_16_hint(dst + OFF_VS + c, vs + c, pol);
            cp_async_16_hint(dst + OFF_VZ + c, vz + c, pol);
        }
        cp_async_mbar_arrive(bar);
        mbar_arrive_expect_tx(bar, TX);
        tma_load_2d_hint(dst, km, kvh * D, pb * kBS, bar, pol);
        tma_load_2d_hint(dst + OFF_V, vm, kvh * (D / 2), pb * kBS, bar, pol);
    }

    static constexpr bool kQ8 = true;
    // quantise staged source row j ([K 2D bytes | V 2D bytes], src dtype) exactly as
    // the write does and put its codes and scales in tile row r
    __device__ __forceinline__ void patch(uint8_t* stg, int r, int j, const uint8_t* buf, int lane,
                                          const AttnParams& p) const {
        constexpr int E = D / 32, LPG = 32 / E;
        const uint16_t* ks = reinterpret_cast<const uint16_t*>(buf + j * 4 * D) + lane * E;
        const uint16_t* vs = reinterpret_cast<const uint16_t*>(buf + j * 4 * D + 2 * D) + lane * E;
        const QuantRow<D> q = p.src_dtype == PKV_BF16 ? quantize_row<__nv_bfloat16, D>(ks, vs)
                                                       : quantize_row<__half, D>(ks, vs);
        // explicit shared-space stores: a generic store here costs the block loop
        // its schedule (measured)
        const uint32_t sa = smem_addr(stg);
        const int kb = lane * E, vb = lane * E / 2;   // this lane's first K byte / V byte in the row
        const uint32_t kd = sa + r * D + 16 * swz<D>(kb >> 4, r) + (kb & 15);
        const uint32_t vd = sa + OFF_V + r * (D / 2) + 16 * swz<D / 2>(vb >> 4, r) + (vb & 15);
        if constexpr (E == 4) {
            sts_u32(kd, q.kpack);
            sts_u16(vd, uint16_t(q.vpack));
        } else {
            sts_u16(kd, uint16_t(q.kpack));
            sts_u8(vd, q.vpack & 0xffu);
        }
        if (lane == 0) sts_u16(sa + OFF_KS + 2 * r, __half_as_ushort(q.ks));
        if (lane % LPG == 0) {
            sts_u16(sa + OFF_VS + 2 * (r * NG + lane / LPG), __half_as_ushort(q.vs));
            sts_u16(sa + OFF_VZ + 2 * (r * NG + lane / LPG), __half_as_ushort(q.vz));
        }
    }

    __device__ __forceinline__ void init(int) {}

    // query column n = head (n / q_len), draft (n % q_len)
    template <bool CASC>
    __device__ __forceinline__ void begin(const AttnParams& p, int s, int kvh, int ctx, int lane) {
        const int g = lane >> 2, t = lane & 3;
        const int G = p.num_heads / p.num_kv_heads, QL = p.q_len, M = G * QL;
        lo_ = visible_lo<CASC>(p, s, ctx);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int n = 8 * nt + g;
            const int h = n < M ? n / QL : 0, j = n < M ? n % QL : 0;
            const int qr = n < M ? query_row<CASC>(p, s, j) : -1;
            const bool valid = qr >= 0;
            const size_t qoff = (size_t(valid ? qr : 0) * p.num_heads + kvh * G + h) * D;
            // this thread's dims t*D/4 .. t*D/4 + D/4 - 1: D/2 contiguous bytes, as 16-byte loads
            uint32_t qw[D / 8];
            const uint4* qv = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.q) + qoff + t * (D / 4));
#pragma unroll
            for (int i = 0; i < D / 32; ++i) {
                const uint4 x = valid ? qv[i] : make_uint4(0u, 0u, 0u, 0u);
                qw[4 * i] = x.x; qw[4 * i + 1] = x.y; qw[4 * i + 2] = x.z; qw[4 * i + 3] = x.w;
            }
            if (p.q_dtype == PKV_BF16) {   // the MMA takes fp16: convert each pair
#pragma unroll
                for (int i = 0; i < D / 8; ++i) {
                    const float2 f = Half16<__nv_bfloat16>::unpack2(qw[i]);
                    qw[i] = pack2<false>(f.x, f.y);
                }
            }
            float qs = 0.f;   // this thread's share of column g's sum of q (in fp16, as the MMA sees it)
#pragma unroll
            for (int kk = 0; kk < NKS; ++kk) {
                qb[nt][kk][0] = qw[2 * kk];       // dims d0, d0 + 1 (d0 = t*D/4 + 4*kk)
                qb[nt][kk][1] = qw[2 * kk + 1];   // dims d0 + 2, d0 + 3
                const float2 f0 = Half16<__half>::unpack2(qw[2 * kk]), f1 = Half16<__half>::unpack2(qw[2 * kk + 1]);
                qs += (f0.x + f0.y) + (f1.x + f1.y);
            }
            qs += __shfl_xor_sync(0xffffffffu, qs, 1);
            qs += __shfl_xor_sync(0xffffffffu, qs, 2);
            // column 2t + e's sum sits in the lanes of g = 2t + e
            kbias[nt][0] = 1152.f * __shfl_sync(0xffffffffu, qs, (2 * t) * 4);
            kbias[nt][1] = 1152.f * __shfl_sync(0xffffffffu, qs, (2 * t + 1) * 4);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int n2 = 8 * nt + 2 * t + e;
                const int j2 = n2 % QL;
                const bool ok2 = n2 < M && query_row<CASC>(p, s, j2) >= 0;
                lim[nt][e] = ok2 ? (CASC ? ctx : max(0, ctx - QL + j2 + 1)) : 0;
                m_run[nt][e] = -INFINITY;
                l_part[nt][e] = 0.f;
            }
#pragma unroll
            for (int mt = 0; mt < 2 * NG; ++mt) o[nt][mt][0] = o[nt][mt][1] = o[nt][mt][2] = o[nt][mt][3] = 0.f;
            cz[nt][0] = cz[nt][1] = cz[nt][2] = cz[nt][3] = 0.f;
        }
        lim_lo_ = INT_MAX;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                if (lim[nt][e] > 0) lim_lo_ = min(lim_lo_, lim[nt][e]);
    }

    __device__ __forceinline__ void block(const uint8_t* stg, int pos0, int ntok, uint8_t*, int lane) {
        const int g = lane >> 2, t = lane & 3;
        const uint32_t stg_a = smem_addr(stg);
        // ------------------------------------------------ S^T = K Q^T (rows = tokens g, g+8)
        uint32_t w[2][NKS];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int row = g + 8 * r;
#pragma unroll
            for (int i = 0; i < D / 64; ++i) {
                const int c = t * (D / 64) + i;
                const uint4 v = *reinterpret_cast<const uint4*>(stg + row * D + 16 * swz<D>(c, row));
                w[r][4 * i] = v.x; w[r][4 * i + 1] = v.y; w[r][4 * i + 2] = v.z; w[r][4 * i + 3] = v.w;
            }
        }
        float sc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
        for (int kk = 0; kk < NKS; ++kk) {
            uint32_t a[4];
            s8x4_to_f16x4_biased(w[0][kk], a[0], a[2]);
            s8x4_to_f16x4_biased(w[1][kk], a[1], a[3]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_f16(sc[nt], a, qb[nt][kk][0], qb[nt][kk][1]);
        }
        // take the codes' bias off: S = sum (c + 1152) q - 1152 sum q
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            sc[nt][0] -= kbias[nt][0];
            sc[nt][1] -= kbias[nt][1];
            sc[nt][2] -= kbias[nt][0];
            sc[nt][3] -= kbias[nt][1];
        }
        // K scale per token, base-2 softmax scale, causal / context mask
        const __half* ksh = reinterpret_cast<const __half*>(stg + OFF_KS);
        const float k0 = __half2float(ksh[g]) * scale_log2_, k1 = __half2float(ksh[g + 8]) * scale_log2_;
        const int pg = pos0 + g, pg8 = pos0 + g + 8;
        if (pos0 >= lo_ && pos0 + kBS <= lim_lo_) {
            // the whole block is visible to every live column of this thread;
            // columns with nothing visible (padding) stay masked
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                sc[nt][0] = lim[nt][0] > 0 ? sc[nt][0] * k0 : -INFINITY;
                sc[nt][1] = lim[nt][1] > 0 ? sc[nt][1] * k0 : -INFINITY;
                sc[nt][2] = lim[nt][0] > 0 ? sc[nt][2] * k1 : -INFINITY;
                sc[nt][3] = lim[nt][1] > 0 ? sc[nt][3] * k1 : -INFINITY;
            }
        } else {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                sc[nt][0] = (pg < lim[nt][0] && pg >= lo_) ? sc[nt][0] * k0 : -INFINITY;
                sc[nt][1] = (pg < lim[nt][1] && pg >= lo_) ? sc[nt][1] * k0 : -INFINITY;
                sc[nt][2] = (pg8 < lim[nt][0] && pg8 >= lo_) ? sc[nt][2] * k1 : -INFINITY;
                sc[nt][3] = (pg8 < lim[nt][1] && pg8 >= lo_) ? sc[nt][3] * k1 : -INFINITY;
            }
        }
        // ------------------------------------------------ online softmax per query column
        float alpha[NT][2];
        bool rescale = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float bm = fmaxf(sc[nt][e], sc[nt][2 + e]);
                bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 4));
                bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 8));
                bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 16));
                const float mn = fmaxf(m_run[nt][e], bm);
                const float mu = (mn == -INFINITY) ? 0.f : mn;
                // nothing accumulated yet (padding columns stay so): no rescale
                alpha[nt][e] = (m_run[nt][e] == -INFINITY) ? 1.f : exp2_ftz(m_run[nt][e] - mu);
                const float p0 = exp2_ftz(sc[nt][e] - mu), p1 = exp2_ftz(sc[nt][2 + e] - mu);
                sc[nt][e] = p0;
                sc[nt][2 + e] = p1;
                l_part[nt][e] = l_part[nt][e] * alpha[nt][e] + (p0 + p1);
                m_run[nt][e] = mn;
                rescale |= alpha[nt][e] != 1.f;
            }
        if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                for (int mt = 0; mt < 2 * NG; ++mt) {
                    o[nt][mt][0] *= alpha[nt][0]; o[nt][mt][2] *= alpha[nt][0];
                    o[nt][mt][1] *= alpha[nt][1]; o[nt][mt][3] *= alpha[nt][1];
                }
                cz[nt][0] *= alpha[nt][0];
                cz[nt][1] *= alpha[nt][1];
            }
        }
        // ------------------------------------------------ P^T operand (tokens 2t.. , query g)
        uint32_t pb[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            pb[nt][0] = movm_trans(pack2<false>(sc[nt][0], sc[nt][1]));
            pb[nt][1] = movm_trans(pack2<false>(sc[nt][2], sc[nt][3]));
        }
        // per-token V scales / zeros of tokens 2t, 2t+1, 2t+8, 2t+9 (all groups);
        // rows past the context hold NaN and are zeroed (their P is 0)
        constexpr int RW = (NG * 2 + 3) / 4;   // 32-bit words per token row
        uint32_t sr[4][RW], zr[4][RW];
        if constexpr (RW == 2) {
            // tokens (2t, 2t+1) and (2t+8, 2t+9): 16 contiguous bytes each
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int tk = 2 * t + 8 * h;
                const uint4 sv = *reinterpret_cast<const uint4*>(stg + OFF_VS + tk * NG * 2);
                const uint4 zv = *reinterpret_cast<const uint4*>(stg + OFF_VZ + tk * NG * 2);
                sr[2 * h][0] = sv.x; sr[2 * h][1] = sv.y; sr[2 * h + 1][0] = sv.z; sr[2 * h + 1][1] = sv.w;
                zr[2 * h][0] = zv.x; zr[2 * h][1] = zv.y; zr[2 * h + 1][0] = zv.z; zr[2 * h + 1][1] = zv.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tk = 2 * t + (i & 1) + 8 * (i >> 1);
                const uint32_t* sp = reinterpret_cast<const uint32_t*>(stg + OFF_VS + tk * NG * 2);
                const uint32_t* zp = reinterpret_cast<const uint32_t*>(stg + OFF_VZ + tk * NG * 2);
#pragma unroll
                for (int q = 0; q < RW; ++q) {
                    sr[i][q] = sp[q];
                    zr[i][q] = zp[q];
                }
            }
        }
        if (ntok < kBS) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int tk = 2 * t + (i & 1) + 8 * (i >> 1);
                if (tk >= ntok) {
#pragma unroll
                    for (int q = 0; q < RW; ++q) sr[i][q] = zr[i][q] = 0u;
                }
            }
        }
        // ------------------------------------------------ O^T += V^T (P^T * s), Z^T P^T
#pragma unroll
        for (int g0 = 0; g0 < NG; g0 += 2) {
            const int mi = lane >> 3, r = lane & 7;
            const int tok = (mi & 1) * 8 + r, c = g0 + (mi >> 1);   // 16-byte chunk = group
            const uint32_t addr = stg_a + OFF_V + tok * (D / 2) + 16 * swz<D / 2>(c, tok);
            uint32_t X[4];
            ldsm_x4_t(addr, X);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int gg = g0 + h;
                const uint32_t xlo = X[2 * h], xhi = X[2 * h + 1];
                // {s[token a][gg], s[token b][gg]} pairs for tokens (2t, 2t+1) and (2t+8, 2t+9)
                const uint32_t sel = (gg & 1) ? 0x7632u : 0x5410u;
                const uint32_t s01 = __byte_perm(sr[0][gg >> 1], sr[1][gg >> 1], sel);
                const uint32_t s89 = __byte_perm(sr[2][gg >> 1], sr[3][gg >> 1], sel);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    uint32_t a[4];
                    a[0] = u4pair_to_f16x2(xlo, i);
                    a[1] = u4pair_to_f16x2(xlo, i + 2);
                    a[2] = u4pair_to_f16x2(xhi, i);
                    a[3] = u4pair_to_f16x2(xhi, i + 2);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma_f16(o[nt][2 * gg + i], a, hmul2_u32(pb[nt][0], s01), hmul2_u32(pb[nt][1], s89));
                }
            }
        }
        {
            // zero points: A rows = groups (row g of this thread, g < NG), k = tokens
            const uint32_t sel = (g & 1) ? 0x7632u : 0x5410u;
            uint32_t z[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) z[i] = (RW > 1 && (g & 2)) ? zr[i][RW - 1] : zr[i][0];
            uint32_t za[4];
            za[0] = g < NG ? __byte_perm(z[0], z[1], sel) : 0u;
            za[1] = 0u;
            za[2] = g < NG ? __byte_perm(z[2], z[3], sel) : 0u;
            za[3] = 0u;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_f16(cz[nt], za, pb[nt][0], pb[nt][1]);
        }
    }

    // add the zero-point term of each group, then sum l over the 8 token lanes
    __device__ __forceinline__ void finish(int lane) {
        const int t = lane & 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int gg = 0; gg < NG; ++gg) {
                const float z0 = __shfl_sync(0xffffffffu, cz[nt][0], gg * 4 + t);
                const float z1 = __shfl_sync(0xffffffffu, cz[nt][1], gg * 4 + t);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    o[nt][2 * gg + i][0] += z0; o[nt][2 * gg + i][2] += z0;
                    o[nt][2 * gg + i][1] += z1; o[nt][2 * gg + i][3] += z1;
                }
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                float l = l_part[nt][e];
                l += __shfl_xor_sync(0xffffffffu, l, 4);
                l += __shfl_xor_sync(0xffffffffu, l, 8);
                l += __shfl_xor_sync(0xffffffffu, l, 16);
                l_part[nt][e] = l;
            }
        }
    }

    // unnormalised rows [M][D] and per-row (m, l) of this warp
    __device__ __forceinline__ void store(float* ob, float* mw, float* lw, int M, int lane) const {
        const int g = lane >> 2, t = lane & 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int q = 8 * nt + 2 * t + e;
                if (q >= M) continue;
#pragma unroll
                for (int gg = 0; gg < NG; ++gg)
                    *reinterpret_cast<float4*>(ob + ob_idx(q, 32 * gg + 4 * g, D)) =
                        make_float4(o[nt][2 * gg][e], o[nt][2 * gg + 1][e], o[nt][2 * gg][2 + e], o[nt][2 * gg + 1][2 + e]);
                if (g == 0) {
                    mw[q] = m_run[nt][e];
                    lw[q] = l_part[nt][e];
                }
            }
    }
};

// ---------------------------------------------------------------- work list

__device__ __forceinline__ int seq_ctx(const AttnParams& p, int s) {
    int c = p.context_lens[s];
    const int cap = p.max_blocks * kBS;
    return c < 0 ? 0 : (c > cap ? cap : c);
}

// First unit of a sequence (blocks / partitions wholly before its first visible
// token are skipped) and its number of units: balanced = blocks; split = partitions.
template <bool CASC>
__device__ __forceinline__ int seq_first_unit(const AttnParams& p, int s, int ctx) {
    const int b = visible_lo<CASC>(p, s, ctx) / kBS;
    return p.mode == kModeBalanced ? b : b / p.partition_blocks;
}
template <bool CASC>
__device__ __forceinline__ long long seq_units(const AttnParams& p, int s, int ctx) {
    const int nb = (ctx + kBS - 1) / kBS;
    const int all = p.mode == kModeBalanced ? nb : (nb + p.partition_blocks - 1) / p.partition_blocks;
    return all - seq_first_unit<CASC>(p, s, ctx);
}

struct Seg {
    int s, kvh, b0, b1, nb, ctx, part;
    long long nu;           // units of this (sequence, kv head) pair
    long long pair_start;   // balanced: the sequence's first unit (block) in the lane's list
    long long cost_base;    // balanced: unit u of this pair sits at cost position u + cost_base
    bool whole;             // the segment is the whole pair
};

// Iterates this CTA's segments in order.  Every warp runs its own copy; all
// lanes of a warp hold the same state.
template <bool CASC>
struct SegIter {
    long long u, u1;
    int kvh;             // split / balanced: the kv head of this CTA's lane
    int s;               // current sequence (split / balanced)
    long long start;     // its first unit
    long long n;         // its units
    int nb, ctx;
    int u_first;         // first unit (block or partition) of s
    int r;               // non-empty sequences before s in the lane's list

    __device__ __forceinline__ void load_seq(const AttnParams& p, int s_, long long start_, int known_ctx = -1) {
        s = s_;
        start = start_;
        if (s < p.num_seqs) {
            ctx = known_ctx >= 0 ? known_ctx : seq_ctx(p, s);
            nb = (ctx + kBS - 1) / kBS;
            u_first = seq_first_unit<CASC>(p, s, ctx);
            n = seq_units<CASC>(p, s, ctx);
        } else {
            ctx = nb = u_first = 0;
            n = 0;
        }
    }

    __device__ __forceinline__ bool next(const AttnParams& p, Seg& g) {
        if (u >= u1) return false;
        if (p.mode == kModeSingle) {
            const int Hkv = p.num_kv_heads;
            g.s = int(u / Hkv);
            g.kvh = int(u % Hkv);
            g.ctx = seq_ctx(p, g.s);
            g.nb = (g.ctx + kBS - 1) / kBS;
            g.b0 = visible_lo<CASC>(p, g.s, g.ctx) / kBS;
            g.b1 = g.nb;
            g.nu = 1;
            g.part = 0;
            g.pair_start = 0;
            g.cost_base = 0;
            g.whole = true;
            u += 1;
            return true;
        }
        while (s < p.num_seqs && u >= start + n) {
            r += (n > 0);
            load_seq(p, s + 1, start + n);
        }
        if (s >= p.num_seqs) {
            u = u1;
            return false;
        }
        const long long k = u - start;
        g.s = s;
        g.kvh = kvh;
        g.nb = nb;
        g.ctx = ctx;
        g.nu = n;
        if (p.mode == kModeBalanced) {
            const long long k1 = (n < k + (u1 - u)) ? n : k + (u1 - u);
            g.b0 = u_first + int(k);
            g.b1 = u_first + int(k1);
            g.part = 0;
            g.pair_start = start;
            g.cost_base = (long long)p.seg_cost * (r + 1);
            g.whole = (k == 0 && k1 == n);
            u += k1 - k;
        } else {
            g.part = u_first + int(k);
            g.b0 = max(g.part * p.partition_blocks, visible_lo<CASC>(p, s, ctx) / kBS);
            g.b1 = min(nb, (g.part + 1) * p.partition_blocks);
            g.pair_start = 0;
            g.cost_base = 0;
            g.whole = false;
            u += 1;
        }
        return true;
    }
};

// Block-wide plan of a split / balanced CTA.  The lane's list holds every
// sequence's units in order.  Balanced mode charges each non-empty sequence
// seg_cost virtual units ahead of its first block (the merge and combine of one
// more segment), then cuts the list's total cost into nlanes equal ranges, so a
// CTA whose range starts a sequence is given fewer blocks.  Unit u of sequence s
// sits at cost position u + seg_cost * (r_s + 1), r_s = non-empty sequences
// before s.  The first sequence's charge lies before every range (a CTA that
// starts with it has no extra segment): CTA k serves cost range
// [seg_cost + k * chunk, seg_cost + (k + 1) * chunk).
struct Plan {
    long long u0, u1, chunk, start0;
    int s0, ctx0, r0;
};

// Plan scratch: red[0 .. warps) holds the block-wide scan's per-warp totals (at
// most 16 warps), red[16 .. 19) this CTA's resolved start / end.
constexpr int kRedSlots = 24;
constexpr int kRedU1 = 16, kRedU0 = 17, kRedStart0 = 18;
constexpr int kRedTl = 20;   // timeline build: this launch's index

// Timeline build (-DPKV_TIMELINE, a separate library that the product never
// loads): thread 0 / lane 0 stamp %globaltimer at fixed points of each CTA's
// run into p.timeline: word 0 counts CTA entries (launch index = count / grid),
// then [launch % kTlLaunches][CTA][kTlWords]: 0 entry, 1 plan done, 2 first
// copies issued (after the grid dependency wait), 3 first block in shared
// memory, 4 + 4k + {0, 1, 2, 3} segment k (< kTlSegs): start, blocks merged,
// piece published, end; 28 segments | combiner bits << 8 | piece bits << 16;
// 29 + k/4: blocks of segment k, 16 bits each.
constexpr int kTlLaunches = 64, kTlCtas = 160, kTlWords = 32, kTlSegs = 6;
#ifdef PKV_TIMELINE
#define PKV_TL_AT(word, value)                                                                              \
    do {                                                                                                    \
        if (p.timeline && blockIdx.x < kTlCtas)                                                             \
            p.timeline[1 + (size_t(tl_launch % kTlLaunches) * kTlCtas + blockIdx.x) * kTlWords + (word)] = \
                (value);                                                                                    \
    } while (0)
#define PKV_TL(word) PKV_TL_AT(word, global_timer_ns())
#else
#define PKV_TL_AT(word, value) \
    do {                       \
    } while (0)
#define PKV_TL(word) PKV_TL_AT(word, 0)
#endif

struct SeqPos {
    int s, ctx;
    long long u, U, C;   // units, first unit, first cost position
};

// One round of nthr sequences from r0: a block-wide scan of (cost << 32 | units)
// gives this thread's sequence its first unit and cost position.
template <bool CASC>
__device__ __forceinline__ SeqPos plan_round(const AttnParams& p, int r0, long long* red,
                                             unsigned long long& base) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    SeqPos sp;
    sp.s = r0 + threadIdx.x;
    sp.ctx = sp.s < p.num_seqs ? seq_ctx(p, sp.s) : 0;
    sp.u = sp.s < p.num_seqs ? seq_units<CASC>(p, sp.s, sp.ctx) : 0;
    const unsigned long long v =
        sp.u > 0 ? ((unsigned long long)(sp.u + p.seg_cost) << 32) | (unsigned long long)sp.u : 0ull;
    unsigned long long incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) red[warp] = (long long)incl;
    __syncthreads();
    unsigned long long before = 0, total = 0;
    for (int w = 0; w < nw; ++w) {
        if (w < warp) before += (unsigned long long)red[w];
        total += (unsigned long long)red[w];
    }
    const unsigned long long excl = base + before + incl - v;
    sp.U = (long long)(excl & 0xffffffffull);
    sp.C = (long long)(excl >> 32);
    base += total;
    __syncthreads();
    return sp;
}

// Where cost positions X0 (this CTA's start) and X1 (its end) fall, if in sp.
__device__ __forceinline__ void plan_resolve(const AttnParams& p, const SeqPos& sp, long long X0, long long X1,
                                             long long* red, int* flag) {
    if (sp.u <= 0) return;
    const long long sc = p.seg_cost, c_end = sp.C + sc + sp.u;
    if (sp.C <= X0 && X0 < c_end) {
        flag[0] = sp.s;
        flag[2] = sp.ctx;
        flag[3] = sc > 0 ? int((sp.C - sp.U) / sc) : 0;
        red[kRedStart0] = sp.U;
        red[kRedU0] = sp.U + max(0ll, X0 - sp.C - sc);
    }
    if (sp.C <= X1 && X1 < c_end) red[kRedU1] = sp.U + max(0ll, X1 - sp.C - sc);
}

template <bool CASC>
__device__ void cta_plan(const AttnParams& p, int lane_idx, int nlanes, long long* red, int* flag, Plan& pl) {
    const int B = p.num_seqs, nthr = blockDim.x;
    unsigned long long base = 0;
    SeqPos mine{};
    for (int r0 = 0; r0 < B; r0 += nthr) mine = plan_round<CASC>(p, r0, red, base);
    const long long total_u = (long long)(base & 0xffffffffull), total_c = (long long)(base >> 32);
    // split mode charges nothing (seg_cost 0)
    const long long span = total_c > p.seg_cost ? total_c - p.seg_cost : 0;
    long long chunk = (span + nlanes - 1) / nlanes;
    if (p.mode == kModeBalanced && chunk < p.min_chunk + p.seg_cost) chunk = p.min_chunk + p.seg_cost;
    if (chunk < 1) chunk = 1;
    const long long X0 = p.seg_cost + lane_idx * chunk, X1 = X0 + chunk;
    if (threadIdx.x == 0) {
        flag[0] = B;         // s0
        flag[2] = 0;         // ctx0
        flag[3] = 0;         // r0
        red[kRedStart0] = 0;   // start0
        red[kRedU0] = total_u;   // u0 (X0 past the end: empty range)
        red[kRedU1] = total_u;   // u1
    }
    __syncthreads();
    if (B <= nthr) {
        plan_resolve(p, mine, X0, X1, red, flag);
    } else {
        base = 0;
        for (int r0 = 0; r0 < B; r0 += nthr) plan_resolve(p, plan_round<CASC>(p, r0, red, base), X0, X1, red, flag);
    }
    __syncthreads();
    pl.chunk = chunk;
    pl.u0 = red[kRedU0];
    pl.u1 = red[kRedU1];
    pl.s0 = flag[0];
    pl.ctx0 = flag[2];
    pl.r0 = flag[3];
    pl.start0 = red[kRedStart0];
}

// ---------------------------------------------------------------- fused decode step: cache writes

// This CTA's share of the step's cache writes (what pkv_reshape_and_cache or
// pkv_quantize_kv does): fp16/bf16 rows as 16-byte chunks, K8/V4 rows by one
// warp each through quantize_row.  Slots < 0 are padding; slots past the pool
// are skipped and flagged.
template <bool Q8, int D>
__device__ void fused_write(const AttnParams& p, int warp, int nwarps, int tid) {
    // Work is dealt out warp by warp across all CTAs (task w goes to warp
    // w / grid of CTA w % grid), so every CTA's share fits in the first TMA
    // round trip instead of a few CTAs starting late.
    const int H = p.num_kv_heads, lane = tid & 31;
    const int64_t pool = int64_t(p.num_blocks) * kBS;
    const int64_t w0 = int64_t(warp) * gridDim.x + blockIdx.x, nw = int64_t(nwarps) * gridDim.x;
    if constexpr (!Q8) {
        // 32 consecutive 16-byte chunks of the [T, H*D*2 bytes] rows per task, four tasks' loads in flight
        const int chunks = H * D * 2 / 16;
        const int64_t total = int64_t(p.num_new) * chunks, ntask = (total + 31) / 32;
        for (int64_t t0 = w0; t0 < ntask; t0 += 4 * nw) {
            uint4 kv[4], vv[4];
            int64_t slot[4], idx[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                idx[u] = (t0 + u * nw) * 32 + lane;
                slot[u] = -1;
                if (t0 + u * nw < ntask && idx[u] < total) {
                    slot[u] = p.slot_mapping[idx[u] / chunks];
                    kv[u] = __ldg(reinterpret_cast<const uint4*>(p.k_new) + idx[u]);
                    vv[u] = __ldg(reinterpret_cast<const uint4*>(p.v_new) + idx[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (slot[u] < 0) continue;
                const int64_t c = idx[u] % chunks;
                if (slot[u] >= pool) {
                    if (c == 0) flag_error(p.err, PKV_DEVERR_OOB_SLOT);
                    continue;
                }
                reinterpret_cast<uint4*>(p.kc)[slot[u] * chunks + c] = kv[u];
                reinterpret_cast<uint4*>(p.vc)[slot[u] * chunks + c] = vv[u];
            }
        }
    } else {
        // one (token, kv head) row per task, quantised by the whole warp
        constexpr int E = D / 32, NG = D / 32, LPG = 32 / E;
        for (int64_t w = w0; w < int64_t(p.num_new) * H; w += nw) {
            const int64_t tok = w / H;
            const int h = int(w - tok * H);
            const int64_t slot = p.slot_mapping[tok];
            if (slot < 0) continue;
            if (slot >= pool) {
                if (lane == 0) flag_error(p.err, PKV_DEVERR_OOB_SLOT);
                continue;
            }
            const int64_t src = (tok * H + h) * D + lane * E;
            const uint16_t* ks = reinterpret_cast<const uint16_t*>(p.k_new) + src;
            const uint16_t* vs = reinterpret_cast<const uint16_t*>(p.v_new) + src;
            const QuantRow<D> q = p.src_dtype == PKV_BF16 ? quantize_row<__nv_bfloat16, D>(ks, vs)
                                                           : quantize_row<__half, D>(ks, vs);
            const int64_t blk = slot / kBS, off = slot - blk * kBS;
            const int64_t row = (blk * kBS + off) * H + h;
            const int64_t meta = (blk * H + h) * kBS + off;
            int8_t* kq = reinterpret_cast<int8_t*>(p.kc) + row * D + lane * E;
            uint8_t* vq = reinterpret_cast<uint8_t*>(p.vc) + row * (D / 2) + lane * (E / 2);
            if constexpr (E == 4) {
                *reinterpret_cast<uint32_t*>(kq) = q.kpack;
                *reinterpret_cast<uint16_t*>(vq) = uint16_t(q.vpack);
            } else {
                *reinterpret_cast<uint16_t*>(kq) = uint16_t(q.kpack);
                *vq = uint8_t(q.vpack);
            }
            if (lane == 0) reinterpret_cast<__half*>(const_cast<void*>(p.k_scale))[meta] = q.ks;
            if (lane % LPG == 0) {
                reinterpret_cast<__half*>(const_cast<void*>(p.v_scale))[meta * NG + lane / LPG] = q.vs;
                reinterpret_cast<__half*>(const_cast<void*>(p.v_zero))[meta * NG + lane / LPG] = q.vz;
            }
        }
    }
}

// ---------------------------------------------------------------- the kernel

template <class Math, bool FUSED, bool CASC>
__global__ void __launch_bounds__((Math::NCW + 1) * 32, 1)
attention_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                 const AttnParams p) {
    constexpr int NCW = Math::NCW;
    extern __shared__ uint8_t smem_raw[];
    // 1 KB aligned (the swizzled tiles need it), and derived from smem_raw by an
    // offset so the compiler still knows every pointer below is shared memory
    // (shared loads, not generic ones)
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const int S = p.stages;
    const int G = p.num_heads / p.num_kv_heads, QL = p.q_len, M = G * QL, D = p.head_dim;
    const int H = p.num_heads, Hkv = p.num_kv_heads;
    // shared-memory layout
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(S) * Math::STAGE);
    uint64_t* empty = full + S;
    int* poison = reinterpret_cast<int*>(empty + S);
    long long* red = reinterpret_cast<long long*>(smem + align_up(S * Math::STAGE + 16 * S + 4 * S, 16));
    int* flag = reinterpret_cast<int*>(red + kRedSlots);
    float* mw = reinterpret_cast<float*>(flag + 4);                  // [NCW][16]
    float* lw = mw + NCW * kMaxRows;                                  // [NCW][16]
    // fused step, g = 1 only: [NCW][16 int64 + 16 int32] slot checks (otherwise
    // they sit in the merge buffer behind the staged rows)
    uint8_t* ck = reinterpret_cast<uint8_t*>(lw + NCW * kMaxRows);
    const bool own_ck = FUSED && !checks_fit(M, QL, D);
    float* ob = reinterpret_cast<float*>(ck + (own_ck ? kCheckBytes * NCW : 0));   // [NCW][M][D], ob_idx order
    uint8_t* scratch = reinterpret_cast<uint8_t*>(ob + size_t(NCW) * M * D);   // [NCW][SCRATCH]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tid = threadIdx.x;

    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        fence_barrier_init();
    }
#ifdef PKV_TIMELINE
    unsigned int tl_launch = 0;
    if (tid == 0) {
        tl_launch = p.timeline ? unsigned(atomicAdd(p.timeline, 1ull) / gridDim.x) : 0u;
        red[kRedTl] = tl_launch;
        PKV_TL(0);
    }
    int tl_seg = 0;
    unsigned long long tl_flags = 0, tl_blocks = 0;
    bool tl_first = true;
#endif

    // ---- this CTA's range of units.  Split / balanced: the grid is Hkv lanes of
    // L CTAs; CTA c serves kv head c % Hkv over range c / Hkv of the lane's list,
    // so CTAs c .. c+Hkv-1 stream the same blocks' head slices side by side and
    // every 2*Hkv*D-byte token row of a block is read from DRAM at one time.
    const int lane_kvh = blockIdx.x % Hkv, lane_idx = blockIdx.x / Hkv, nlanes = gridDim.x / Hkv;
    if (CASC || p.wait_first) grid_dep_wait();   // the plan reads what the previous kernel wrote
    Plan pl;
    if (p.mode == kModeSingle) {
        const long long total = (long long)p.num_seqs * Hkv;
        pl.chunk = (total + gridDim.x - 1) / gridDim.x;
        pl.u0 = blockIdx.x * pl.chunk;
        pl.u1 = pl.u0 + pl.chunk < total ? pl.u0 + pl.chunk : total;
        pl.s0 = 0;
        pl.ctx0 = -1;
        pl.r0 = 0;
        pl.start0 = 0;
        __syncthreads();
    } else {
        cta_plan<CASC>(p, lane_idx, nlanes, red, flag, pl);
    }
    const long long chunk = pl.chunk;
    // Except in a cascade pass or with wait_first, everything above read only the
    // launch's inputs (context lengths), which no kernel of this library writes; what follows
    // waits for the previous kernel of the stream before it reads the cache or
    // writes anything.
#ifdef PKV_TIMELINE
    tl_launch = unsigned(red[kRedTl]);   // the plan's barriers made it visible
    if (tid == 0) PKV_TL(1);
#endif
    if (tid == 0) grid_dep_launch();

    SegIter<CASC> it;
    it.u = pl.u0;
    it.u1 = pl.u0 < pl.u1 ? pl.u1 : pl.u0;
    it.kvh = lane_kvh;
    it.r = pl.r0;
    if (p.mode != kModeSingle) it.load_seq(p, pl.s0, pl.start0, pl.ctx0);

    if (warp == NCW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&k_map);
            prefetch_tensormap(&v_map);
        }
        // Up to `grp` consecutive blocks are issued per pass, one per lane: each
        // lane waits for its own stage, reads its own block-table entry and
        // issues its own copies, so the per-block chain (wait, expect_tx, TMA)
        // of different blocks overlaps.  grp <= S: the previous use of every
        // stage touched in a pass was issued by an earlier pass.
        const int grp = S < Math::kIssueGroup ? S : Math::kIssueGroup;
        int issued = 0;   // blocks issued by this CTA
        bool waited = false;
        Seg sg;
        while (it.next(p, sg)) {
            const int bt_seq = CASC ? p.item_seq[sg.s] : sg.s;   // cascade: an item reads its lending member's table
            const int32_t* bt = p.block_tables + size_t(bt_seq) * p.max_blocks;
            const int n = sg.b1 - sg.b0;
            for (int i0 = 0; i0 < n; i0 += grp) {
                if (lane < grp && i0 + lane < n) {
                    int pb = bt[sg.b0 + i0 + lane];   // block tables: an input, read before the wait
                    if (!waited) {
                        grid_dep_wait();
                        waited = true;
#ifdef PKV_TIMELINE
                        if (lane == 0) PKV_TL(2);
#endif
                    }
                    const int j = issued + lane;
                    const int st = j % S;
                    const int use = j / S;
                    if (use > 0 && !mbar_wait(&empty[st], uint32_t((use - 1) & 1)))
                        flag_error(p.err, PKV_DEVERR_TIMEOUT);
                    const int bad = (pb < 0 || pb >= p.num_blocks);
                    if (bad) {
                        flag_error(p.err, PKV_DEVERR_OOB_BLOCK);
                        pb = 0;   // load a valid block; the consumer masks it out
                    }
                    poison[st] = bad;
                    Math::issue(smem + size_t(st) * Math::STAGE, &k_map, &v_map, p, sg.kvh, pb, &full[st]);
                }
                issued += min(grp, n - i0);
                __syncwarp();
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    constexpr int CT = NCW * 32;   // consumer threads
    grid_dep_wait();
    // context longer than its table: flagged once per sequence
    for (int s = blockIdx.x * CT + tid; s < p.num_seqs; s += gridDim.x * CT)
        if (p.context_lens[s] > p.max_blocks * kBS) flag_error(p.err, PKV_DEVERR_CAPACITY);
    constexpr int kPer = (kMaxRows * 128 / 4 + CT - 1) / CT;   // float4 outputs per thread, at most
    // fused decode step: write this CTA's share of the new tokens; the attention
    // below takes in-place tokens from k_new / v_new (patched into the tiles),
    // so no CTA has to wait for another's write
    if constexpr (FUSED) fused_write<Math::kQ8, Math::kD>(p, warp, NCW, tid);
    // balanced mode: sequences with nothing visible still get their zero rows
    // (cascade: an empty partial in the sequence's own slot)
    if (p.mode == kModeBalanced) {
        if constexpr (CASC) {
            for (int s = p.num_items + blockIdx.x; s < p.num_seqs; s += gridDim.x)
                if (seq_units<CASC>(p, s, seq_ctx(p, s)) == 0)
                    for (int h = tid; h < H; h += CT) {
                        const size_t pi = (size_t(query_row<CASC>(p, s, 0)) * H + h) * p.max_partitions;
                        p.max_logits[pi] = -INFINITY;
                        p.exp_sums[pi] = 0.f;
                    }
        } else {
            for (int s = blockIdx.x; s < p.num_seqs; s += gridDim.x)
                if (seq_ctx(p, s) == 0)
                    for (int i = tid; i < QL * H * D; i += CT)
                        store_out(p.out, p.out_dtype, size_t(s) * QL * H * D + i, 0.f);
        }
    }

    Math mth;
    mth.init(lane);
    if constexpr (Math::kTensor) mth.scale_log2_ = p.scale_log2;
    uint8_t* my_scratch = scratch + warp * Math::SCRATCH;
    int jbase = 0;   // blocks of this CTA before the current segment
    Seg sg;
    while (it.next(p, sg)) {
        const int n = sg.b1 - sg.b0;
#ifdef PKV_TIMELINE
        if (tid == 0 && tl_seg < kTlSegs) PKV_TL(4 + 4 * tl_seg);
#endif
        mth.template begin<CASC>(p, sg.s, sg.kvh, sg.ctx, lane);
        // Fused step: the warp that will consume a block holding new positions
        // [ctx - q_len, ctx) prefetches those rows from k_new / v_new into its
        // merge buffer (free until the merge) with cp.async, and their slot
        // checks into registers; it patches them into the tile when the block
        // arrives.  New row j is "in place" when its slot is that of its own
        // position: then the tile takes k_new / v_new instead of the cache.
        uint8_t* staged = reinterpret_cast<uint8_t*>(ob + size_t(warp) * M * D);
        // the rows' slot_mapping entries and block-table entries: this warp's check area
        int64_t* st_slot = reinterpret_cast<int64_t*>(own_ck ? ck + warp * kCheckBytes : staged + QL * 4 * D);
        int32_t* st_pb = reinterpret_cast<int32_t*>(st_slot + kMaxRows);
        const int new0 = sg.ctx - QL;   // position of new row 0
        bool owner = false;
        if (FUSED && sg.ctx > 0) {
            const int t0 = max(new0, 0) / kBS, t1 = (sg.ctx - 1) / kBS;
            for (int b = max(t0, sg.b0); b <= min(t1, sg.b1 - 1); ++b)
                owner |= ((jbase + b - sg.b0) % NCW) == warp;
            if (owner) {
                const size_t tok0 = size_t(sg.s) * QL;
                if (lane < QL) {
                    if (tok0 + lane < size_t(p.num_new) && new0 + lane >= 0) {
                        cp_async_8(st_slot + lane, p.slot_mapping + tok0 + lane);
                        cp_async_4(st_pb + lane, p.block_tables + size_t(sg.s) * p.max_blocks + (new0 + lane) / kBS);
                    } else {
                        st_slot[lane] = -1;
                        st_pb[lane] = -1;
                    }
                }
                constexpr int CHK = Math::kD * 2 / 16;   // 16-byte chunks of a source row
                for (int c = lane; c < QL * 2 * CHK; c += 32) {
                    const int jj = c / (2 * CHK), r = c - jj * (2 * CHK);
                    if (tok0 + jj < size_t(p.num_new)) {
                        const uint8_t* src = static_cast<const uint8_t*>(r < CHK ? p.k_new : p.v_new) +
                                             ((tok0 + jj) * Hkv + sg.kvh) * size_t(Math::kD) * 2 + 16 * (r % CHK);
                        cp_async_16(staged + jj * 4 * Math::kD + 16 * r, src);
                    }
                }
                cp_async_commit();
            }
        }
        const int i_first = (warp - jbase % NCW + NCW) % NCW;
        // stage and phase of this warp's blocks, advanced by NCW per block (S is
        // a multiple of NCW) instead of a division per block
        int st = (jbase + i_first) % S;
        uint32_t phase = uint32_t((jbase + i_first) / S) & 1u;
        for (int i = i_first; i < n; i += NCW) {
            const bool ok = mbar_wait(&full[st], phase);
#ifdef PKV_TIMELINE
            if (tl_first && warp == 0 && lane == 0) PKV_TL(3);
            tl_first = false;
#endif
            if (!ok && lane == 0) flag_error(p.err, PKV_DEVERR_TIMEOUT);
            const int b = sg.b0 + i;
            int ntok = (b == sg.nb - 1) ? sg.ctx - b * kBS : kBS;
            if (!ok || poison[st]) ntok = 0;
            bool patched = false;
            if (FUSED && owner && ntok > 0 && new0 + QL > b * kBS && new0 < (b + 1) * kBS) {
                cp_async_wait_all();
                __syncwarp();
                const int pos_l = new0 + lane;
                const int64_t my_slot = lane < QL ? st_slot[lane] : -1;
                const int my_pb = lane < QL ? st_pb[lane] : -1;
                const bool in_place = lane < QL && my_slot >= 0 && pos_l >= 0 && pos_l >= visible_lo<CASC>(p, sg.s, sg.ctx) &&
                                      my_pb >= 0 && my_pb < p.num_blocks &&
                                      my_slot == int64_t(my_pb) * kBS + pos_l % kBS;
                const uint32_t mask = __ballot_sync(0xffffffffu, in_place);
                for (int jj = 0; jj < QL; ++jj) {
                    const int pos = new0 + jj;
                    if (((mask >> jj) & 1u) && pos >= b * kBS && pos < (b + 1) * kBS) {
                        mth.patch(smem + size_t(st) * Math::STAGE, pos - b * kBS, jj, staged, lane, p);
                        patched = true;
                    }
                }
                __syncwarp();
            }
            if (ntok > 0) mth.block(smem + size_t(st) * Math::STAGE, b * kBS, ntok, my_scratch, lane);
            // generic writes into a stage the TMA refills: order them before the refill
            if (FUSED && patched) fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            st += NCW;
            if (st >= S) {
                st -= S;
                phase ^= 1u;
            }
        }
        jbase += n;
        mth.finish(lane);

        // ------------------------------------------------ merge the warps' states for this segment
        mth.store(ob + size_t(warp) * M * D, mw + warp * kMaxRows, lw + warp * kMaxRows, M, lane);
        named_barrier_sync(1, CT);
#ifdef PKV_TIMELINE
        if (tid == 0 && tl_seg < kTlSegs) PKV_TL(4 + 4 * tl_seg + 1);
#endif
        // Every shared-memory read of the merge comes before the first global
        // store: a store can wait behind this SM's queue of TMA reads, and a
        // later shared load issued behind it would wait as long.  Each thread
        // works out its row's segment max, the warps' weights 2^(m_w - max) and
        // the sum itself (no second barrier).
        const int n4 = (M * D) >> 2;
        float4 res[kPer];
        float resM[kPer], resL[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i4 = tid + k * CT;
            float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
            float Mx = -INFINITY, L = 0.f;
            if (i4 < n4) {
                const int m = (i4 << 2) / D, d = (i4 << 2) - m * D;
                float mwv[NCW];
#pragma unroll
                for (int w2 = 0; w2 < NCW; ++w2) {
                    mwv[w2] = mw[w2 * kMaxRows + m];
                    Mx = fmaxf(Mx, mwv[w2]);
                }
#pragma unroll
                for (int w2 = 0; w2 < NCW; ++w2) {
                    const float f = (mwv[w2] == -INFINITY) ? 0.f : exp2f(mwv[w2] - Mx);
                    L = fmaf(lw[w2 * kMaxRows + m], f, L);
                    const float4 v = *reinterpret_cast<const float4*>(ob + size_t(w2) * M * D + ob_idx(m, d, D));
                    O.x = fmaf(v.x, f, O.x);
                    O.y = fmaf(v.y, f, O.y);
                    O.z = fmaf(v.z, f, O.z);
                    O.w = fmaf(v.w, f, O.w);
                }
            }
            res[k] = O;
            resM[k] = Mx;
            resL[k] = L;
        }
        const int pair = sg.s * Hkv + sg.kvh;
        const bool piece = (p.mode == kModeBalanced) && !sg.whole;
        // piece slot: unique because (lane_idx + s) grows along a lane's pieces
        const int slot = (lane_idx + sg.s) * Hkv + sg.kvh;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int i4 = tid + k * CT;
            if (i4 >= n4) continue;
            const int m = (i4 << 2) / D, d = (i4 << 2) - m * D;
            const float L = resL[k], Mx = resM[k];
            const int h = m / QL, jq = m - (m / QL) * QL;
            const int qrow = query_row<CASC>(p, sg.s, jq);
            if (CASC && qrow < 0) continue;   // a cascade item's padding column
            const size_t row = size_t(qrow);
            const int hg = sg.kvh * G + h;
            if (piece) {
                reinterpret_cast<float4*>(p.part_o + (size_t(slot) * kMaxRows + m) * D)[d >> 2] = res[k];
                if (d == 0)
                    reinterpret_cast<float2*>(p.part_ml)[size_t(slot) * kMaxRows + m] = make_float2(Mx, L);
            } else {
                // a row whose sum is not positive (no visible token, or a NaN read
                // from a poisoned slot) is written as zeros
                const bool live = L > 0.f;
                const float inv = live ? 1.f / L : 0.f;
                const float4 o = live ? make_float4(res[k].x * inv, res[k].y * inv, res[k].z * inv, res[k].w * inv)
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
                if (CASC || p.mode == kModeSplit) {
                    // cascade: an item's partial goes to its members' slot part_offset
                    const int slot_p = sg.part + ((CASC && sg.s < p.num_items) ? p.part_offset : 0);
                    const size_t pi = (row * H + hg) * p.max_partitions + slot_p;
                    reinterpret_cast<float4*>(p.tmp_out + pi * D)[d >> 2] = o;
                    if (d == 0) {
                        p.max_logits[pi] = (L > 0.f) ? Mx * kLn2 : -INFINITY;
                        p.exp_sums[pi] = L;
                    }
                } else {
                    store_out4(p.out, p.out_dtype, (row * H + hg) * D + d, o);
                }
            }
        }
        if (piece) {
            // The last piece of a pair to finish combines all of them (no
            // waiting).  Publication: every thread's partial stores, the barrier,
            // then the count by thread 0 with release semantics at gpu scope (the
            // barrier makes the other threads' stores part of what it releases).
            named_barrier_sync(1, CT);
            const int c_lo = int((sg.pair_start + sg.cost_base - p.seg_cost) / chunk),
                      c_hi = int((sg.pair_start + sg.nu - 1 + sg.cost_base - p.seg_cost) / chunk);
            const int np = c_hi - c_lo + 1;
            if (tid == 0) {
                // release: this CTA's partial stores (ordered by the barrier);
                // acquire: the other pieces' partials before our loads
                const int prev = atomic_add_acq_rel_gpu(&p.counters[pair], 1);
                flag[1] = (prev == np - 1) ? 1 : 0;
            }
            named_barrier_sync(1, CT);
#ifdef PKV_TIMELINE
            if (tid == 0 && tl_seg < kTlSegs) {
                PKV_TL(4 + 4 * tl_seg + 2);
                tl_flags |= (1ull << (16 + tl_seg)) | (flag[1] ? (1ull << (8 + tl_seg)) : 0ull);
            }
#endif
            if (flag[1]) {
                // Pieces hold unnormalised sums relative to their own max m_c:
                // O = sum_c 2^(m_c - M) O_c, L = sum_c 2^(m_c - M) l_c.  The pieces'
                // (m, l) and O slices are loaded eight at a time, all in flight
                // together, and folded in by an online rescale in piece order (so
                // the result does not depend on which CTA combines); this CTA's own
                // piece comes from its registers, not from memory.
                const int own = lane_idx - c_lo;
                constexpr int kFly = 8;
#pragma unroll
                for (int k = 0; k < kPer; ++k) {
                    const int i4 = tid + k * CT;
                    if (i4 >= n4) break;
                    const int m = (i4 << 2) / D, d = (i4 << 2) - m * D;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    float Mr = -INFINITY, Lr = 0.f;
                    for (int c0 = 0; c0 < np; c0 += kFly) {
                        float2 ml[kFly];
                        float4 v[kFly];
#pragma unroll
                        for (int u = 0; u < kFly; ++u) {
                            ml[u] = make_float2(-INFINITY, 0.f);
                            v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                            const int c = c0 + u;
                            if (c == own) {
                                ml[u] = make_float2(resM[k], resL[k]);
                                v[u] = res[k];
                            } else if (c < np) {
                                const size_t sl = size_t((c_lo + c + sg.s) * Hkv + sg.kvh) * kMaxRows;
                                ml[u] = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + sl + m);
                                v[u] = __ldcg(reinterpret_cast<const float4*>(p.part_o + sl * D) + i4);
                            }
                        }
                        float Mn = Mr;
#pragma unroll
                        for (int u = 0; u < kFly; ++u)
                            if (ml[u].y > 0.f) Mn = fmaxf(Mn, ml[u].x);
                        const float a = (Mr == -INFINITY) ? 0.f : exp2f(Mr - Mn);
                        acc.x *= a; acc.y *= a; acc.z *= a; acc.w *= a;
                        Lr *= a;
#pragma unroll
                        for (int u = 0; u < kFly; ++u) {
                            const float f = (ml[u].y > 0.f) ? exp2f(ml[u].x - Mn) : 0.f;
                            acc.x = fmaf(f, v[u].x, acc.x);
                            acc.y = fmaf(f, v[u].y, acc.y);
                            acc.z = fmaf(f, v[u].z, acc.z);
                            acc.w = fmaf(f, v[u].w, acc.w);
                            Lr = fmaf(f, ml[u].y, Lr);
                        }
                        Mr = Mn;
                    }
                    const float L = Lr;
                    const bool live = L > 0.f;
                    const float inv = live ? 1.f / L : 0.f;
                    const int h = m / QL, jq = m - (m / QL) * QL;
                    const float4 o = live ? make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                    if constexpr (CASC) {
                        // the pair's combined partial into its slot (items: part_offset)
                        const int qrow = query_row<CASC>(p, sg.s, jq);
                        if (qrow < 0) continue;
                        const size_t pi = (size_t(qrow) * H + sg.kvh * G + h) * p.max_partitions +
                                          (sg.s < p.num_items ? p.part_offset : 0);
                        reinterpret_cast<float4*>(p.tmp_out + pi * D)[d >> 2] = o;
                        if (d == 0) {
                            p.max_logits[pi] = live ? Mr * kLn2 : -INFINITY;
                            p.exp_sums[pi] = L;
                        }
                    } else {
                        store_out4(p.out, p.out_dtype, ((size_t(sg.s) * QL + jq) * H + sg.kvh * G + h) * D + d, o);
                    }
                }
                if (tid == 0) p.counters[pair] = 0;   // ready for the next launch
            }
        }
        named_barrier_sync(1, CT);   // the merge buffers are reused by the next segment
#ifdef PKV_TIMELINE
        if (tid == 0) {
            if (tl_seg < kTlSegs) {
                PKV_TL(4 + 4 * tl_seg + 3);
                if (tl_seg < 4) tl_blocks |= (unsigned long long)(n & 0xffff) << (16 * tl_seg);
            }
            ++tl_seg;
            PKV_TL_AT(28, tl_flags | (unsigned long long)(tl_seg < 255 ? tl_seg : 255));
            PKV_TL_AT(29, tl_blocks);
        }
#endif
    }
}

template <class Math, bool FUSED>
int smem_bytes(int stages, int M, int QL, int D) {
    constexpr int NCW = Math::NCW;
    return stages * Math::STAGE + 16 * stages + 4 * stages + 16 + kRedSlots * 8 + 16 + 2 * NCW * kMaxRows * 4 +
           (FUSED && !checks_fit(M, QL, D) ? NCW * kCheckBytes : 0) + NCW * M * D * 4 + NCW * Math::SCRATCH + 1024 + 64;
}

template <class Math, bool FUSED, bool CASC>
cudaError_t launch_math(AttnParams p, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t stream) {
    static int num_sms = 0;
    if (num_sms == 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    const int M = (p.num_heads / p.num_kv_heads) * p.q_len;
    const int base = smem_bytes<Math, FUSED>(0, M, p.q_len, p.head_dim);
    int stages = (kSmemLimit - base) / (Math::STAGE + 20);
    if (stages > 9 * Math::NCW) stages = 9 * Math::NCW;
    stages = stages / Math::NCW * Math::NCW;   // every stage always belongs to the same consumer warp
    if (stages < Math::NCW) return cudaErrorInvalidConfiguration;
    p.stages = stages;
    if (p.mode == kModeBalanced) p.seg_cost = Math::kSegCost;
    const int smem = smem_bytes<Math, FUSED>(stages, M, p.q_len, p.head_dim);
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attention_kernel<Math, FUSED, CASC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemLimit);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int cap = num_sms < kMaxGrid ? num_sms : kMaxGrid;
    int grid;
    if (p.mode == kModeSingle) {
        const long long pairs = (long long)p.num_seqs * p.num_kv_heads;
        grid = pairs < cap ? int(pairs < 1 ? 1 : pairs) : cap;
    } else {
        // Hkv lanes of L CTAs each (at least one lane)
        int L = cap / p.num_kv_heads;
        if (L < 1) L = 1;
        const long long lane_units = (long long)p.num_seqs * p.max_blocks;   // upper bound of a lane's list
        if (lane_units < L) L = int(lane_units < 1 ? 1 : lane_units);
        grid = L * p.num_kv_heads;
    }
    return launch_kernel(attention_kernel<Math, FUSED, CASC>, dim3(grid), dim3((Math::NCW + 1) * 32), size_t(smem),
                         stream, km, vm, p);
}

template <typename T, int D, bool FUSED>
cudaError_t dispatch_cc(const AttnParams& p, int gqa, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t st) {
    // group sizes 1 and 2 (larger groups run the tensor-core math)
    switch (gqa) {
        case 1: return launch_math<CcMath<T, D, 1>, FUSED, false>(p, km, vm, st);
        case 2: return launch_math<CcMath<T, D, 2>, FUSED, false>(p, km, vm, st);
        default: return cudaErrorInvalidValue;
    }
}

// Math for the cache kind, head_dim, group size and q_len, then launch.  The
// cascade pass takes the tensor-core math (an item has several query rows per
// kv head; the sequences' own entries share its instantiation).  The choice is
// attention_uses_tensor_cores(), the predicate the host also builds the tensor
// maps from: the tensor-core maths issue 3-D tile copies (fp16/bf16) or
// swizzled row copies (K8/V4) that only their own maps describe.
template <bool FUSED, bool CASC>
cudaError_t launch_attention_impl(const AttnParams& p, int cache_kind, int gqa, const CUtensorMap& km,
                                  const CUtensorMap& vm, cudaStream_t stream) {
    if (attention_uses_tensor_cores(cache_kind, p.q_len, gqa, CASC)) {
        switch (cache_kind) {
            case PKV_CACHE_K8V4: {
                const bool narrow = (p.num_heads / p.num_kv_heads) * p.q_len <= 8;
                if (p.head_dim == 128)
                    return narrow ? launch_math<TqMath<128, 1>, FUSED, CASC>(p, km, vm, stream)
                                  : launch_math<TqMath<128, 2>, FUSED, CASC>(p, km, vm, stream);
                return narrow ? launch_math<TqMath<64, 1>, FUSED, CASC>(p, km, vm, stream)
                              : launch_math<TqMath<64, 2>, FUSED, CASC>(p, km, vm, stream);
            }
            case PKV_CACHE_BF16:
                if ((p.num_heads / p.num_kv_heads) * p.q_len <= 8)
                    return p.head_dim == 128 ? launch_math<TtMath<PKV_CACHE_BF16, 128>, FUSED, CASC>(p, km, vm, stream)
                                             : launch_math<TtMath<PKV_CACHE_BF16, 64>, FUSED, CASC>(p, km, vm, stream);
                return p.head_dim == 128 ? launch_math<TcMath<PKV_CACHE_BF16, 128>, FUSED, CASC>(p, km, vm, stream)
                                         : launch_math<TcMath<PKV_CACHE_BF16, 64>, FUSED, CASC>(p, km, vm, stream);
            default:
                if ((p.num_heads / p.num_kv_heads) * p.q_len <= 8)
                    return p.head_dim == 128 ? launch_math<TtMath<PKV_CACHE_F16, 128>, FUSED, CASC>(p, km, vm, stream)
                                             : launch_math<TtMath<PKV_CACHE_F16, 64>, FUSED, CASC>(p, km, vm, stream);
                return p.head_dim == 128 ? launch_math<TcMath<PKV_CACHE_F16, 128>, FUSED, CASC>(p, km, vm, stream)
                                         : launch_math<TcMath<PKV_CACHE_F16, 64>, FUSED, CASC>(p, km, vm, stream);
        }
    }
    if constexpr (!CASC) {
        if (cache_kind == PKV_CACHE_BF16)
            return p.head_dim == 128 ? dispatch_cc<__nv_bfloat16, 128, FUSED>(p, gqa, km, vm, stream)
                                     : dispatch_cc<__nv_bfloat16, 64, FUSED>(p, gqa, km, vm, stream);
        return p.head_dim == 128 ? dispatch_cc<__half, 128, FUSED>(p, gqa, km, vm, stream)
                                 : dispatch_cc<__half, 64, FUSED>(p, gqa, km, vm, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

}  // namespace pkv
