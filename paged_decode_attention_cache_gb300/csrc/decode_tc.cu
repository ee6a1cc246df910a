// decode_tc.cu -- paged attention on tensor cores (mma.sync m16n8k16, fp32
// accumulate) for the two cases whose per-block work is a small dense
// contraction:
//   * the speculative verify block: q_len > 1 draft tokens per sequence, each
//     causally masked among the drafts [mlxcel manual "KV Cache",
//     §"Matrix-Absorbed MLA Decode" (a speculative verify block) and
//     §"Speculative Rewind"]; g heads x q_len drafts = up to 16 query rows per
//     (sequence, kv head) share every K/V block;
//   * the mixed-precision K8/V4 cache [metalworking "The KV Cache", §"The K/V
//     asymmetry"], read without an intermediate dequantised copy [MTPLX "How
//     the Paged KV Cache Works in MTPLX", §"TurboQuant Fast Path": quantised
//     attention without intermediate dequantization steps]: the int8 / int4
//     codes are turned into exact fp16 integers in registers and fed to the
//     MMA, the per-token K scale multiplies the scores, the per-group V scale
//     multiplies P, and the V zero-point term sum_t p_t z_t is added on CUDA
//     cores.
//
// Layout of one CTA (grid = partition x kv head x sequence): warp 4 is the
// producer (TMA tile loads + 1-D bulk copies of the quantiser metadata into an
// S-stage mbarrier ring); warps 0-3 each take whole 16-token blocks:
//   QK^T: A = 16 query rows (row m = head (m / q_len), draft (m % q_len)),
//         B = the block's 16 keys as two n-tiles of 8 tokens;
//   online softmax on the accumulator fragments (rows g and g+8 per lane);
//   PV:   A = P (re-packed accumulator fragments), B = V via ldmatrix.trans.
// Tiles arrive TMA-swizzled (128B / 64B / 32B patterns by row size) so every
// ldmatrix / 128-bit shared load is bank-conflict free.  The warps' states are
// merged through shared memory at the end, as in the CUDA-core kernel.
#include "pkv_device.cuh"
#include "pkv_internal.h"

namespace pkv {

namespace {

constexpr int kBS = 16;
constexpr int kNCW = 4;
constexpr int kThreads = (kNCW + 1) * 32;

constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int KIND, int D>
struct TC {
    static constexpr bool Q8 = KIND == PKV_CACHE_K8V4;
    static constexpr int NG = D / 32;                    // V groups per row
    static constexpr int NKS = D / 16;                   // k-steps of QK
    static constexpr int NNT = D / 8;                    // n-tiles of PV
    static constexpr int KROW = Q8 ? D : 2 * D;          // bytes of one K row
    static constexpr int VROW = Q8 ? D / 2 : 2 * D;
    static constexpr int KT = kBS * KROW;                // K tile bytes
    static constexpr int VT = kBS * VROW;
    static constexpr int KS = Q8 ? kBS * 2 : 0;          // k_scale bytes per block
    static constexpr int VS = Q8 ? kBS * NG * 2 : 0;     // v_scale (and v_zero) bytes per block
    static constexpr int OFF_V = align_up(KT, 1024);
    static constexpr int OFF_KS = OFF_V + align_up(VT, 16);
    static constexpr int OFF_VS = OFF_KS + KS;
    static constexpr int OFF_VZ = OFF_VS + VS;
    static constexpr int TX = KT + VT + KS + 2 * VS;     // bytes landing per stage
    static constexpr int STAGE = align_up(OFF_VZ + VS, 1024);
    static constexpr int S = (65536 / STAGE) < 2 ? 2 : 65536 / STAGE;
    static constexpr int RING = S * STAGE;
    static constexpr int OBUF = kNCW * 16 * D * 4;       // merge buffer, aliases the ring
    static constexpr int OFF_BAR = RING > OBUF ? RING : OBUF;
    static constexpr int OFF_POISON = OFF_BAR + 2 * S * 8;
    static constexpr int OFF_MW = align_up(OFF_POISON + 4 * S, 16);
    static constexpr int OFF_LW = OFF_MW + kNCW * 16 * 4;
    static constexpr int SMEM = OFF_LW + kNCW * 16 * 4 + 1024;   // + slack to align the base
    static_assert(OFF_V % 1024 == 0 && STAGE % 1024 == 0, "swizzled tiles need 1 KB alignment");
};

// Physical 16-byte chunk of logical chunk c in row t of a TMA tile whose rows
// are W bytes long, loaded with the W-byte swizzle (W = 32, 64 or 128).
template <int W>
__device__ __forceinline__ int swz(int c, int t) {
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

// Four int8 codes (one 32-bit word, code e in byte e) -> two fp16x2 holding the
// exact integers: flip the sign bit (c + 128 in 0..255), splice each byte under
// the fp16 exponent of 1024 (0x64xx = 1024 + byte), subtract 1152.
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

// Nibble i of both 16-bit halves of w -> fp16x2 of the exact integers 0..15.
__device__ __forceinline__ uint32_t u4pair_to_f16x2(uint32_t w, int i) {
    const uint32_t x = ((w >> (4 * i)) & 0x000F000Fu) | 0x64006400u;   // 1024 + code
    const __half2 bias = __halves2half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400));
    __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&x), bias);
    return *reinterpret_cast<uint32_t*>(&h);
}

template <int KIND, int D>
__global__ void __launch_bounds__(kThreads, 2)
decode_tc_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                 const AttnParams p) {
    using C = TC<KIND, D>;
    constexpr bool Q8 = C::Q8;
    constexpr bool BF = (KIND == PKV_CACHE_BF16);     // operand type of the fp16/bf16 path
    constexpr int S = C::S;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* empty = full + S;
    int* poison = reinterpret_cast<int*>(smem + C::OFF_POISON);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int part = blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
    const bool split = p.tmp_out != nullptr;
    const int H = p.num_heads, G = p.num_heads / p.num_kv_heads, QL = p.q_len, M = G * QL;

    int ctx = p.context_lens[s];
    const int cap = p.max_blocks * kBS;
    if (ctx > cap) {
        if (part == 0 && threadIdx.x == 0) flag_error(p.err, PKV_DEVERR_CAPACITY);
        ctx = cap;
    }
    if (ctx < 0) ctx = 0;
    const int nblk_seq = (ctx + kBS - 1) / kBS;
    const int b0 = part * p.partition_blocks;
    const int nblk = min(b0 + p.partition_blocks, nblk_seq) - b0;

    if (nblk <= 0) {
        if (!split && part == 0)
            for (int i = threadIdx.x; i < M * D; i += kThreads) {
                const int m = i / D, d = i % D, h = m / QL, j = m % QL;
                store_out(p.out, p.out_dtype, ((size_t(s) * QL + j) * H + kvh * G + h) * D + d, 0.f);
            }
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

    if (warp == kNCW) {
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
                        pb = 0;
                    }
                    poison[st] = bad;
                    uint8_t* dst = smem + st * C::STAGE;
                    mbar_arrive_expect_tx(&full[st], C::TX);
                    if constexpr (Q8) {
                        // byte-addressed maps: x is the byte offset of this kv head in a token row
                        tma_load_2d(dst, &k_map, kvh * D, pb * kBS, &full[st]);
                        tma_load_2d(dst + C::OFF_V, &v_map, kvh * (D / 2), pb * kBS, &full[st]);
                        const size_t meta = size_t(pb) * p.num_kv_heads + kvh;
                        bulk_load(dst + C::OFF_KS, reinterpret_cast<const uint8_t*>(p.k_scale) + meta * C::KS, C::KS,
                                  &full[st]);
                        bulk_load(dst + C::OFF_VS, reinterpret_cast<const uint8_t*>(p.v_scale) + meta * C::VS, C::VS,
                                  &full[st]);
                        bulk_load(dst + C::OFF_VZ, reinterpret_cast<const uint8_t*>(p.v_zero) + meta * C::VS, C::VS,
                                  &full[st]);
                    } else {
#pragma unroll
                        for (int b = 0; b < D / 64; ++b) {   // 128-byte boxes (64 dims) with the 128B swizzle
                            tma_load_2d(dst + b * 2048, &k_map, kvh * D * 2 + b * 128, pb * kBS, &full[st]);
                            tma_load_2d(dst + C::OFF_V + b * 2048, &v_map, kvh * D * 2 + b * 128, pb * kBS, &full[st]);
                        }
                    }
                }
                __syncwarp();
            }
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    const int g = lane >> 2, tid = lane & 3;
    // query rows g and g+8 of the 16-row tile; visible limit of each
    int lim[2];
    uint32_t qa[C::NKS][4];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int m = g + 8 * r;
        const bool valid = m < M;
        const int h = valid ? m / QL : 0, j = valid ? m % QL : 0;
        lim[r] = valid ? max(0, ctx - QL + j + 1) : 0;
        const size_t qoff = ((size_t(s) * QL + j) * H + kvh * G + h) * D;
#pragma unroll
        for (int kk = 0; kk < C::NKS; ++kk) {
            uint32_t lo = 0, hi = 0;
            if (valid) {
                if constexpr (Q8) {
                    // lane's dims for k-step kk: tid*D/4 + 4kk + {0,1 | 2,3}
                    const int d0 = tid * (D / 4) + 4 * kk;
                    const float q0 = load_q(p.q, p.q_dtype, qoff + d0), q1 = load_q(p.q, p.q_dtype, qoff + d0 + 1);
                    const float q2 = load_q(p.q, p.q_dtype, qoff + d0 + 2), q3 = load_q(p.q, p.q_dtype, qoff + d0 + 3);
                    lo = pack2<false>(q0, q1);
                    hi = pack2<false>(q2, q3);
                } else {
                    const uint32_t* qw = reinterpret_cast<const uint32_t*>(p.q);
                    lo = qw[(qoff + 16 * kk + 2 * tid) / 2];
                    hi = qw[(qoff + 16 * kk + 8 + 2 * tid) / 2];
                }
            }
            qa[kk][r] = lo;
            qa[kk][2 + r] = hi;
        }
    }
    float o[C::NNT][4];
#pragma unroll
    for (int n = 0; n < C::NNT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float zacc[2][C::NG];
#pragma unroll
    for (int gg = 0; gg < C::NG; ++gg) zacc[0][gg] = zacc[1][gg] = 0.f;

    for (int j = warp; j < nblk; j += kNCW) {
        const int st = j % S;
        const bool ok = mbar_wait(&full[st], (j / S) & 1);
        if (!ok && lane == 0) flag_error(p.err, PKV_DEVERR_TIMEOUT);
        const int pos0 = (b0 + j) * kBS;
        int ntok = min(kBS, ctx - pos0);
        if (!ok || poison[st]) ntok = 0;
        if (ntok > 0) {
            const uint8_t* stg = smem + st * C::STAGE;
            const uint32_t stg_a = smem_addr(stg);
            float sc[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
            // ------------------------------------------------ S = Q K^T
            if constexpr (Q8) {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const int t = nt * 8 + g;
                    uint32_t w[C::NKS];
#pragma unroll
                    for (int i = 0; i < D / 64; ++i) {
                        const int c = tid * (D / 64) + i;
                        const uint4 v = *reinterpret_cast<const uint4*>(stg + t * D + 16 * swz<D>(c, t));
                        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
                    }
#pragma unroll
                    for (int kk = 0; kk < C::NKS; ++kk) {
                        uint32_t b0, b1;
                        s8x4_to_f16x4(w[kk], b0, b1);
                        mma_f16(sc[nt], qa[kk], b0, b1);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const __half2 ks2 = *reinterpret_cast<const __half2*>(stg + C::OFF_KS + (nt * 8 + 2 * tid) * 2);
                    const float2 ks = __half22float2(ks2);
                    const float k0 = ks.x * p.scale_log2, k1 = ks.y * p.scale_log2;
                    sc[nt][0] *= k0; sc[nt][1] *= k1; sc[nt][2] *= k0; sc[nt][3] *= k1;
                }
            } else {
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
                    for (int kp = 0; kp < C::NKS / 2; ++kp) {
                        const int mi = lane >> 3, r = lane & 7;
                        const int t = nt * 8 + r, c = 4 * kp + mi;           // 8-dim chunk c
                        const uint32_t addr = stg_a + (c >> 3) * 2048 + t * 128 + 16 * swz<128>(c & 7, t);
                        uint32_t R[4];
                        ldsm_x4(addr, R);
                        mma16816<BF>(sc[nt], qa[2 * kp], R[0], R[1]);
                        mma16816<BF>(sc[nt], qa[2 * kp + 1], R[2], R[3]);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) sc[nt][e] *= p.scale_log2;
            }
            // ------------------------------------------------ mask + online softmax (rows g, g+8)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int pos = pos0 + nt * 8 + 2 * tid + (e & 1);
                    if (!(pos < lim[e >> 1])) sc[nt][e] = -INFINITY;
                }
            float alpha[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                float bm = fmaxf(fmaxf(sc[0][2 * r], sc[0][2 * r + 1]), fmaxf(sc[1][2 * r], sc[1][2 * r + 1]));
                bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 1));
                bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, 2));
                const float mn = fmaxf(m_run[r], bm);
                const float mu = (mn == -INFINITY) ? 0.f : mn;
                alpha[r] = exp2f(m_run[r] - mu);
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
                for (int n = 0; n < C::NNT; ++n) {
                    o[n][0] *= alpha[0]; o[n][1] *= alpha[0];
                    o[n][2] *= alpha[1]; o[n][3] *= alpha[1];
                }
#pragma unroll
                for (int gg = 0; gg < C::NG; ++gg) {
                    zacc[0][gg] *= alpha[0];
                    zacc[1][gg] *= alpha[1];
                }
            }
            // ------------------------------------------------ O += P V
            if constexpr (Q8) {
                // the lane's four tokens: 2tid, 2tid+1 (n-tile 0) and 8+2tid, 9+2tid (n-tile 1)
                const int tk[4] = {2 * tid, 2 * tid + 1, 8 + 2 * tid, 9 + 2 * tid};
                float sv[4][C::NG], zv[4][C::NG];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const bool valid = tk[i] < ntok;   // past the context: NaN metadata, keep it out of the MMA
                    const __half* vs = reinterpret_cast<const __half*>(stg + C::OFF_VS) + tk[i] * C::NG;
                    const __half* vz = reinterpret_cast<const __half*>(stg + C::OFF_VZ) + tk[i] * C::NG;
#pragma unroll
                    for (int gg = 0; gg < C::NG; ++gg) {
                        sv[i][gg] = valid ? __half2float(vs[gg]) : 0.f;
                        zv[i][gg] = valid ? __half2float(vz[gg]) : 0.f;
                    }
                }
                // V codes of the lane's tokens, one 16-bit word (4 dims) per (token, group) column g
                uint32_t X[C::NG], Y[C::NG];
#pragma unroll
                for (int g0 = 0; g0 < C::NG; g0 += 2) {
                    const int mi = lane >> 3, r = lane & 7;
                    const int t = (mi & 1) * 8 + r, c = g0 + (mi >> 1);
                    const uint32_t addr = stg_a + C::OFF_V + t * (D / 2) + 16 * swz<D / 2>(c, t);
                    uint32_t R[4];
                    ldsm_x4_t(addr, R);
                    X[g0] = R[0]; Y[g0] = R[1]; X[g0 + 1] = R[2]; Y[g0 + 1] = R[3];
                }
#pragma unroll
                for (int gg = 0; gg < C::NG; ++gg) {
                    uint32_t a[4];
                    a[0] = pack2<false>(sc[0][0] * sv[0][gg], sc[0][1] * sv[1][gg]);
                    a[1] = pack2<false>(sc[0][2] * sv[0][gg], sc[0][3] * sv[1][gg]);
                    a[2] = pack2<false>(sc[1][0] * sv[2][gg], sc[1][1] * sv[3][gg]);
                    a[3] = pack2<false>(sc[1][2] * sv[2][gg], sc[1][3] * sv[3][gg]);
                    zacc[0][gg] += sc[0][0] * zv[0][gg] + sc[0][1] * zv[1][gg] + sc[1][0] * zv[2][gg] +
                                   sc[1][1] * zv[3][gg];
                    zacc[1][gg] += sc[0][2] * zv[0][gg] + sc[0][3] * zv[1][gg] + sc[1][2] * zv[2][gg] +
                                   sc[1][3] * zv[3][gg];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        mma_f16(o[4 * gg + i], a, u4pair_to_f16x2(X[gg], i), u4pair_to_f16x2(Y[gg], i));
                }
            } else {
                uint32_t a[4];
                a[0] = pack2<BF>(sc[0][0], sc[0][1]);
                a[1] = pack2<BF>(sc[0][2], sc[0][3]);
                a[2] = pack2<BF>(sc[1][0], sc[1][1]);
                a[3] = pack2<BF>(sc[1][2], sc[1][3]);
                // V rows past the context may hold anything (NaN): zero them in the operand
                const uint32_t m01 = (2 * tid < ntok ? 0x0000ffffu : 0u) | (2 * tid + 1 < ntok ? 0xffff0000u : 0u);
                const uint32_t m23 = (8 + 2 * tid < ntok ? 0x0000ffffu : 0u) | (9 + 2 * tid < ntok ? 0xffff0000u : 0u);
#pragma unroll
                for (int np = 0; np < C::NNT / 2; ++np) {
                    const int mi = lane >> 3, r = lane & 7;
                    const int t = (mi & 1) * 8 + r, c = 2 * np + (mi >> 1);   // 8-dim chunk = n-tile
                    const uint32_t addr = stg_a + C::OFF_V + (c >> 3) * 2048 + t * 128 + 16 * swz<128>(c & 7, t);
                    uint32_t R[4];
                    ldsm_x4_t(addr, R);
                    if (ntok < kBS) {
                        R[0] &= m01; R[1] &= m23; R[2] &= m01; R[3] &= m23;
                    }
                    mma16816<BF>(o[2 * np], a, R[0], R[1]);
                    mma16816<BF>(o[2 * np + 1], a, R[2], R[3]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }

    if constexpr (Q8) {
        // V zero-point term: sum over the row's tokens of p_t * z_t, same for every dim of a group
#pragma unroll
        for (int gg = 0; gg < C::NG; ++gg)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                float z = zacc[r][gg];
                z += __shfl_xor_sync(0xffffffffu, z, 1);
                z += __shfl_xor_sync(0xffffffffu, z, 2);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    o[4 * gg + i][2 * r] += z;
                    o[4 * gg + i][2 * r + 1] += z;
                }
            }
    }

    // ------------------------------------------------------------ merge the warps
    named_barrier_sync(1, kNCW * 32);   // every stage consumed: the ring is free for the merge buffer
    float* ob = reinterpret_cast<float*>(smem);
    float* mw = reinterpret_cast<float*>(smem + C::OFF_MW);
    float* lw = reinterpret_cast<float*>(smem + C::OFF_LW);
#pragma unroll
    for (int n = 0; n < C::NNT; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int m = g + 8 * (e >> 1), col = 2 * tid + (e & 1);
            const int d = Q8 ? 32 * (n >> 2) + 4 * col + (n & 3) : 8 * n + col;
            ob[(warp * 16 + m) * D + d] = o[n][e];
        }
    if (tid == 0) {
        mw[warp * 16 + g] = m_run[0];
        mw[warp * 16 + g + 8] = m_run[1];
        lw[warp * 16 + g] = l_run[0];
        lw[warp * 16 + g + 8] = l_run[1];
    }
    named_barrier_sync(1, kNCW * 32);
    for (int idx = threadIdx.x; idx < M * D; idx += kNCW * 32) {
        const int m = idx / D, d = idx % D;
        float Mx = -INFINITY;
#pragma unroll
        for (int w2 = 0; w2 < kNCW; ++w2) Mx = fmaxf(Mx, mw[w2 * 16 + m]);
        float L = 0.f, O = 0.f;
        if (Mx != -INFINITY) {
#pragma unroll
            for (int w2 = 0; w2 < kNCW; ++w2) {
                const float mm = mw[w2 * 16 + m];
                if (mm != -INFINITY) {
                    const float f = exp2f(mm - Mx);
                    L = fmaf(lw[w2 * 16 + m], f, L);
                    O = fmaf(ob[(w2 * 16 + m) * D + d], f, O);
                }
            }
        }
        const int h = m / QL, jq = m % QL;
        const size_t row = size_t(s) * QL + jq;
        const int hg = kvh * G + h;
        const float val = (L > 0.f) ? O / L : 0.f;
        if (split) {
            const size_t pi = (row * H + hg) * p.max_partitions + part;
            p.tmp_out[pi * D + d] = val;
            if (d == 0) {
                p.max_logits[pi] = (L > 0.f) ? Mx * kLn2 : -INFINITY;
                p.exp_sums[pi] = L;
            }
        } else {
            store_out(p.out, p.out_dtype, (row * H + hg) * D + d, val);
        }
    }
}

template <int KIND, int D>
cudaError_t launch_one(const AttnParams& p, const CUtensorMap& km, const CUtensorMap& vm, int grid_parts,
                       cudaStream_t stream) {
    using C = TC<KIND, D>;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e =
            cudaFuncSetAttribute(decode_tc_kernel<KIND, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    dim3 grid(grid_parts, p.num_kv_heads, p.num_seqs);
    decode_tc_kernel<KIND, D><<<grid, kThreads, C::SMEM, stream>>>(km, vm, p);
    return cudaGetLastError();
}

}  // namespace

bool decode_tc_supported(int cache_kind, int head_dim, int gqa, int q_len) {
    return (cache_kind == PKV_CACHE_F16 || cache_kind == PKV_CACHE_BF16 || cache_kind == PKV_CACHE_K8V4) &&
           (head_dim == 64 || head_dim == 128) && (gqa == 1 || gqa == 2 || gqa == 4 || gqa == 8) && q_len >= 1 &&
           gqa * q_len <= 16;
}

cudaError_t launch_decode_tc(const AttnParams& p, int cache_kind, int gqa, const CUtensorMap& k_map,
                             const CUtensorMap& v_map, int grid_parts, cudaStream_t stream) {
    (void)gqa;
    switch (cache_kind) {
        case PKV_CACHE_K8V4:
            return p.head_dim == 128 ? launch_one<PKV_CACHE_K8V4, 128>(p, k_map, v_map, grid_parts, stream)
                                     : launch_one<PKV_CACHE_K8V4, 64>(p, k_map, v_map, grid_parts, stream);
        case PKV_CACHE_BF16:
            return p.head_dim == 128 ? launch_one<PKV_CACHE_BF16, 128>(p, k_map, v_map, grid_parts, stream)
                                     : launch_one<PKV_CACHE_BF16, 64>(p, k_map, v_map, grid_parts, stream);
        default:
            return p.head_dim == 128 ? launch_one<PKV_CACHE_F16, 128>(p, k_map, v_map, grid_parts, stream)
                                     : launch_one<PKV_CACHE_F16, 64>(p, k_map, v_map, grid_parts, stream);
    }
}

}  // namespace pkv
