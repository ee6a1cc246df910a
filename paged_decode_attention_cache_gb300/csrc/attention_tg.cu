// attention_tg.cu -- balanced attention over a K8/V4 cache (head_dim 128) on
// the 5th-generation tensor cores: tcgen05.mma with shared-memory operands and
// tensor-memory accumulators.
//
// What it computes is what the other attention kernels compute (for every query
// row, softmax over the visible tokens of scale * q . k, times v), with k and v
// the dequantised codes [metalworking "The KV Cache", §"The K/V asymmetry":
// K int8 with a per-token scale, V 4-bit with a scale and zero per group].
//
// Work is cut exactly as in the balanced schedule of attention_impl.cuh (same
// plan, same pieces and workspace slots, same last-arriver combine), but a
// segment is streamed in chunks of 8 blocks (128 tokens), and one CTA keeps a
// single softmax state per query row:
//   producer warp   TMA loads of each block's codes into a ring of stages; the
//                   stage of chunk slot i is (8 * chunk + i) mod S, so every
//                   stage always serves the same dequant warp;
//   8 dequant warps warp i expands slot i of every chunk: K codes to exact fp16
//                   integers, V codes to fp16 values c * s + z (one fused
//                   multiply-add), into the chunk's fp16 tiles in the 128-byte
//                   swizzled layout the MMA reads (two chunks in flight); tokens
//                   that do not exist (past the context, a bad block id, an empty
//                   slot of the last chunk) become zero rows;
//   MMA warp        one thread issues, per chunk, S^T = K Q^T (M = 128 tokens,
//                   N = 16 query columns, K = 128 dims) and, once the softmax
//                   has written P, O^T = V^T P^T (M = 128 dims, N = 16, K = 128
//                   tokens), each into its own tensor-memory buffer, completing
//                   on mbarriers (tcgen05.commit);
//   softmax warps   warps 0-3 own tensor-memory lanes 0-127: thread t reads the
//                   scores of token t, applies the token's K scale, the softmax
//                   scale and the masks, takes the chunk's column maxima across
//                   the four warps, writes P (fp16) and keeps its partial sums;
//                   then it reads row t of the chunk's O^T (one head dim) and
//                   folds it into its running output with the online rescale.
// The V tile stores each 8-dim group in the order {0,4,1,5,2,6,3,7} (the order
// the 4-bit expansion produces), so tensor-memory lane t of O^T holds head dim
// (t & ~7) | perm(t & 7).
#include "attention_impl.cuh"
#include "pkv_umma.cuh"

namespace pkv {

namespace {

constexpr int TG_D = 128;
constexpr int TG_CH = 8;                  // blocks per chunk
constexpr int TG_TOK = TG_CH * kBS;       // tokens per chunk (the MMA's M)
constexpr int TG_NDQ = 8;                 // dequant warps: one chunk slot each
constexpr int TG_WG = 4;                  // softmax warps (tensor-memory lanes 0..127)
constexpr int TG_MMA_WARP = TG_WG + TG_NDQ;
constexpr int TG_PROD_WARP = TG_MMA_WARP + 1;
constexpr int TG_THREADS = (TG_PROD_WARP + 1) * 32;
constexpr int TG_COMPUTE_WARPS = TG_MMA_WARP;   // warps that share the fused step's writes
constexpr int TG_N = 16;                  // the MMA's N: query columns, padded
constexpr int TG_TMEM_COLS = 64;          // S^T [2] at columns 0 / 16, O^T [2] at 32 / 48
constexpr int TG_OPER = TG_TOK * TG_D * 2;   // one fp16 chunk tile: 32 KB
constexpr int TG_QT = TG_N * TG_D * 2;       // the Q tile or one P tile: 4 KB
constexpr int TG_KST = kBS * TG_D;           // K codes of a block: 16 rows of 128 bytes
constexpr int TG_VST = kBS * TG_D / 2;       // V codes: 16 rows of 64 bytes
constexpr int TG_MST = 288;                  // k scales (32 B), v scales (128 B), v zeros (128 B)
constexpr int TG_M_KS = 0, TG_M_VS = 32, TG_M_VZ = 160;
constexpr int TG_OFF_KH = 0;                 // K tiles [2]
constexpr int TG_OFF_VH = 2 * TG_OPER;       // V tiles [2]
constexpr int TG_OFF_Q = 4 * TG_OPER;
constexpr int TG_OFF_P = TG_OFF_Q + TG_QT;   // P tiles [2]
constexpr int TG_OFF_RING = TG_OFF_P + 2 * TG_QT;
constexpr int TG_NBAR = 15;   // chunk full, K tile free, V tile free, S full, P full, O full, O empty [2 each], Q ready
static_assert(TG_OFF_RING % 1024 == 0, "the code ring needs 1 KB alignment");

// instruction descriptors: S^T = K Q^T (both K-major), O^T = V^T P^T (V MN-major)
constexpr uint32_t TG_IDESC_S = umma_idesc_f16(TG_TOK, TG_N, false, false);
constexpr uint32_t TG_IDESC_O = umma_idesc_f16(TG_D, TG_N, true, false);

// bytes of the small arrays after the ring
__host__ __device__ constexpr int tg_small_bytes(int S) {
    return align_up((2 * S + TG_NBAR) * 8, 16) + align_up(4 * S, 16) + 2 * TG_TOK * 4 + 2 * TG_CH * 4 +
           3 * TG_WG * TG_N * 4 + kRedSlots * 8 + 16 + 16 + 16;
}
__host__ __device__ constexpr int tg_smem_bytes(int S) {
    return TG_OFF_RING + S * (TG_KST + TG_VST + TG_MST) + tg_small_bytes(S) + 1024;
}

// head dim held at row t of the V tile / tensor-memory lane t of O^T
__device__ __forceinline__ int tg_dim_of(int t) { return (t & ~7) | ((t & 1) ? 4 + ((t & 7) >> 1) : ((t & 7) >> 1)); }

// TMA of one block's codes (K 2 KB, V 1 KB; 128- and 64-byte swizzled rows) and
// cp.async of its scales and zeros, all completing on `bar`.
__device__ __forceinline__ void tg_issue(uint8_t* kst, uint8_t* vst, uint8_t* mst, const CUtensorMap* km,
                                         const CUtensorMap* vm, const AttnParams& p, int kvh, int pb,
                                         uint64_t* bar) {
    const size_t meta = size_t(pb) * p.num_kv_heads + kvh;
    const uint8_t* ks = reinterpret_cast<const uint8_t*>(p.k_scale) + meta * 32;
    const uint8_t* vs = reinterpret_cast<const uint8_t*>(p.v_scale) + meta * 128;
    const uint8_t* vz = reinterpret_cast<const uint8_t*>(p.v_zero) + meta * 128;
    cp_async_16(mst + TG_M_KS, ks);
    cp_async_16(mst + TG_M_KS + 16, ks + 16);
#pragma unroll
    for (int c = 0; c < 128; c += 16) {
        cp_async_16(mst + TG_M_VS + c, vs + c);
        cp_async_16(mst + TG_M_VZ + c, vz + c);
    }
    cp_async_mbar_arrive(bar);
    mbar_arrive_expect_tx(bar, TG_KST + TG_VST);
    tma_load_2d(kst, km, kvh * TG_D, pb * kBS, bar);
    tma_load_2d(vst, vm, kvh * (TG_D / 2), pb * kBS, bar);
}

// Quantise new token row j of sequence s's step (k_new / v_new, this warp's kv
// head) exactly as the write does and put its codes and scales in row r of the
// stage.
__device__ __forceinline__ void tg_patch(uint8_t* kst, uint8_t* vst, uint8_t* mst, int r, size_t tok, int kvh,
                                         int lane, const AttnParams& p) {
    constexpr int E = TG_D / 32, LPG = 32 / E;
    const size_t src = (tok * p.num_kv_heads + kvh) * TG_D + lane * E;
    const uint16_t* ks = reinterpret_cast<const uint16_t*>(p.k_new) + src;
    const uint16_t* vs = reinterpret_cast<const uint16_t*>(p.v_new) + src;
    const QuantRow<TG_D> q = p.src_dtype == PKV_BF16 ? quantize_row<__nv_bfloat16, TG_D>(ks, vs)
                                                      : quantize_row<__half, TG_D>(ks, vs);
    const int kb = lane * E, vb = lane * E / 2;
    sts_u32(smem_addr(kst) + r * TG_D + 16 * swz<TG_D>(kb >> 4, r) + (kb & 15), q.kpack);
    sts_u16(smem_addr(vst) + r * (TG_D / 2) + 16 * swz<TG_D / 2>(vb >> 4, r) + (vb & 15), uint16_t(q.vpack));
    if (lane == 0) sts_u16(smem_addr(mst) + TG_M_KS + 2 * r, __half_as_ushort(q.ks));
    if (lane % LPG == 0) {
        sts_u16(smem_addr(mst) + TG_M_VS + 2 * (r * 4 + lane / LPG), __half_as_ushort(q.vs));
        sts_u16(smem_addr(mst) + TG_M_VZ + 2 * (r * 4 + lane / LPG), __half_as_ushort(q.vz));
    }
}

// Expand one block (16 tokens) into rows 16 * slot .. 16 * slot + 15 of the
// chunk's K tile; rows >= ntok become zeros.  Lane l takes token l / 2 and the
// head dims 64 * (l % 2) .. + 63 (one 64-dim column block of the tile).  The K
// codes become exact fp16 integers; the per-token scale is applied to the scores.
__device__ __forceinline__ void tg_dequant_k(const uint8_t* kst, uint8_t* kh, int slot, int ntok, int lane) {
    const int r = lane & 15, hb = lane >> 4;
    const int R = slot * kBS + r;   // row in the chunk tiles
    const bool live = r < ntok;
    uint4 w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c = hb * 4 + i;   // 16-code chunk of the 128-byte row
        w[i] = live ? *reinterpret_cast<const uint4*>(kst + r * TG_D + 16 * swz<TG_D>(c, r)) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t h[8];
        s8x4_to_f16x4(w[i].x, h[0], h[1]);
        s8x4_to_f16x4(w[i].y, h[2], h[3]);
        s8x4_to_f16x4(w[i].z, h[4], h[5]);
        s8x4_to_f16x4(w[i].w, h[6], h[7]);
        if (!live) {
#pragma unroll
            for (int e = 0; e < 8; ++e) h[e] = 0u;
        }
        // dims 16c .. 16c + 15: fp16 chunks 2i, 2i + 1 of column block hb
        *reinterpret_cast<uint4*>(kh + sw128_off(R, 64 * hb + 16 * i, TG_TOK)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(kh + sw128_off(R, 64 * hb + 16 * i + 8, TG_TOK)) = make_uint4(h[4], h[5], h[6], h[7]);
    }
}

// The same block's V codes into the chunk's V tile: two 32-dim groups per lane,
// c * s + z in fp16, the dims of each 8-dim run stored in the order
// {0,4,1,5,2,6,3,7}.
__device__ __forceinline__ void tg_dequant_v(const uint8_t* vst, const uint8_t* mst, uint8_t* vh, int slot, int ntok,
                                             int lane) {
    const int r = lane & 15, hb = lane >> 4;
    const int R = slot * kBS + r;
    const bool live = r < ntok;
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
        const int g = 2 * hb + gi;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        __half2 s2 = __half2half2(__ushort_as_half(0)), z2 = s2;
        if (live) {
            w = *reinterpret_cast<const uint4*>(vst + r * (TG_D / 2) + 16 * swz<TG_D / 2>(g, r));
            s2 = __half2half2(*reinterpret_cast<const __half*>(mst + TG_M_VS + 2 * (r * 4 + g)));
            z2 = __half2half2(*reinterpret_cast<const __half*>(mst + TG_M_VZ + 2 * (r * 4 + g)));
        }
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t h[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t c2 = u4pair_to_f16x2(ww[q], i);   // (dim i, dim 4 + i) as exact fp16 integers
                __half2 c;
                memcpy(&c, &c2, 4);
                const __half2 v = __hfma2(c, s2, z2);
                memcpy(&h[i], &v, 4);
            }
            if (!live) h[0] = h[1] = h[2] = h[3] = 0u;
            *reinterpret_cast<uint4*>(vh + sw128_off(R, 64 * hb + 32 * gi + 8 * q, TG_TOK)) =
                make_uint4(h[0], h[1], h[2], h[3]);
        }
    }
}

// A bounded mbarrier wait that gives up at once after any wait of this CTA has
// timed out (then the CTA runs to its end without waiting, flagging the error),
// so a stalled pipeline costs one wait limit, not one per chunk.
__device__ __forceinline__ bool tg_wait(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* err) {
    if (*abort) return false;
    if (mbar_wait(bar, parity)) return true;
    *abort = 1;
    flag_error(err, PKV_DEVERR_TIMEOUT);
    return false;
}

template <int NV, bool FUSED>
__global__ void __launch_bounds__(TG_THREADS, 1)
attention_tg_kernel(const __grid_constant__ CUtensorMap k_map, const __grid_constant__ CUtensorMap v_map,
                    const AttnParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.stages;   // a multiple of TG_CH
    const int G = p.num_heads / p.num_kv_heads, QL = p.q_len, MQ = G * QL;
    const int H = p.num_heads, Hkv = p.num_kv_heads;
    constexpr int D = TG_D;
    uint8_t* kring = smem + TG_OFF_RING;
    uint8_t* vring = kring + size_t(S) * TG_KST;
    uint8_t* mring = vring + size_t(S) * TG_VST;
    uint8_t* sm = mring + size_t(S) * TG_MST;
    uint64_t* full = reinterpret_cast<uint64_t*>(sm);
    uint64_t* empty = full + S;
    uint64_t* cb = empty + S;   // chunk barriers
    uint64_t* chunk_full = cb;
    uint64_t* k_free = cb + 2;    // the K tile's S MMA is done
    uint64_t* v_free = cb + 4;    // the chunk's O MMA is done (V tile, P, K scales, mask)
    uint64_t* s_full = cb + 6;
    uint64_t* p_full = cb + 8;
    uint64_t* o_full = cb + 10;
    uint64_t* o_empty = cb + 12;
    uint64_t* q_ready = cb + 14;
    int* poison = reinterpret_cast<int*>(sm + align_up((2 * S + TG_NBAR) * 8, 16));
    float* kscale = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(poison) + align_up(4 * S, 16));   // [2][128]
    uint32_t* tmask = reinterpret_cast<uint32_t*>(kscale + 2 * TG_TOK);                                   // [2][8]
    float* colx = reinterpret_cast<float*>(tmask + 2 * TG_CH);                                            // [2][4][16]
    float* lsum = colx + 2 * TG_WG * TG_N;                                                                // [4][16]
    long long* red = reinterpret_cast<long long*>(lsum + TG_WG * TG_N);
    int* flag = reinterpret_cast<int*>(red + kRedSlots);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(flag + 4);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    if (tid == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&chunk_full[i], TG_NDQ);
            mbar_init(&k_free[i], 1);
            mbar_init(&v_free[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], TG_WG);
            mbar_init(&o_full[i], 1);
            mbar_init(&o_empty[i], TG_WG);
        }
        mbar_init(q_ready, 1);
        *abort = 0;
        fence_barrier_init();
    }
    if (warp == TG_MMA_WARP) {
        tmem_alloc(smem_addr(tmem_slot), TG_TMEM_COLS);
        tmem_relinquish();
        tc_fence_before_sync();
    }

    // ---- this CTA's range: the balanced plan of attention_impl.cuh
    const int lane_kvh = blockIdx.x % Hkv, lane_idx = blockIdx.x / Hkv, nlanes = gridDim.x / Hkv;
    if (p.wait_first) grid_dep_wait();   // the plan reads what the previous kernel wrote
    Plan pl;
    cta_plan<false>(p, lane_idx, nlanes, red, flag, pl);   // ends on __syncthreads
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const long long chunk = pl.chunk;
    if (tid == 0) grid_dep_launch();

    SegIter<false> it;
    it.u = pl.u0;
    it.u1 = pl.u0 < pl.u1 ? pl.u1 : pl.u0;
    it.kvh = lane_kvh;
    it.r = pl.r0;
    it.load_seq(p, pl.s0, pl.start0, pl.ctx0);

    if (warp == TG_PROD_WARP) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&k_map);
            prefetch_tensormap(&v_map);
        }
        long long ch = 0;
        bool waited = false;
        Seg sg;
        while (it.next(p, sg)) {
            const int32_t* bt = p.block_tables + size_t(sg.s) * p.max_blocks;
            const int nch = (sg.b1 - sg.b0 + TG_CH - 1) / TG_CH;
            for (int c = 0; c < nch; ++c, ++ch) {
                if (lane < TG_CH) {
                    const int b = sg.b0 + c * TG_CH + lane;
                    const bool has = b < sg.b1;
                    int pb = has ? bt[b] : 0;   // block tables: an input, read before the wait
                    if (!waited) {
                        grid_dep_wait();
                        waited = true;
                    }
                    const long long j = ch * TG_CH + lane;
                    const int st = int(j % S);
                    const long long use = j / S;
                    if (use > 0) tg_wait(&empty[st], uint32_t((use - 1) & 1), abort, p.err);
                    if (has) {
                        const int bad = (pb < 0 || pb >= p.num_blocks);
                        if (bad) {
                            flag_error(p.err, PKV_DEVERR_OOB_BLOCK);
                            pb = 0;   // load a valid block; its rows are zeroed and masked
                        }
                        poison[st] = bad;
                        tg_issue(kring + size_t(st) * TG_KST, vring + size_t(st) * TG_VST, mring + size_t(st) * TG_MST,
                                 &k_map, &v_map, p, sg.kvh, pb, &full[st]);
                    } else {
                        poison[st] = 1;   // an empty slot of the segment's last chunk
                        mbar_arrive(&full[st]);
                    }
                }
                __syncwarp();
            }
        }
    } else if (warp == TG_MMA_WARP) {
        // ------------------------------------------------------------ MMA issue
        // Order within a segment: S(0), then per chunk c: S(c + 1) (as soon as its
        // tiles are in), then O(c) (once the softmax has written P(c)), so the
        // scores of the next chunk are ready when the softmax warps finish this
        // one.  S(c + 1) reuses the tensor-memory buffer of S(c - 1), which the
        // softmax released before O(c - 1) was issued.  The first S of a segment
        // comes after the previous segment's last O: it reads the segment's query
        // tile, which the softmax warps write once they have folded that O.
        if (lane == 0) {
            const uint32_t kh0 = smem_addr(smem + TG_OFF_KH), vh0 = smem_addr(smem + TG_OFF_VH);
            const uint32_t qt = smem_addr(smem + TG_OFF_Q), pt0 = smem_addr(smem + TG_OFF_P);
            long long nxt = 0;   // chunks whose S has been issued
            int segno = -1;      // segments started
            bool new_seg = false;
            Seg sg;
            int c_in = 0, nch = 0;   // position in the current segment's chunks
            auto advance = [&]() -> bool {   // is there a next chunk (and does it start a segment)?
                while (c_in >= nch) {
                    if (!it.next(p, sg)) return false;
                    nch = (sg.b1 - sg.b0 + TG_CH - 1) / TG_CH;
                    c_in = 0;
                    if (nch > 0) new_seg = true;
                }
                return true;
            };
            auto issue_s = [&]() {
                if (new_seg) {
                    ++segno;
                    tg_wait(q_ready, uint32_t(segno & 1), abort, p.err);
                    new_seg = false;
                }
                const long long ch = nxt;
                const int buf = int(ch & 1);
                tg_wait(&chunk_full[buf], uint32_t((ch >> 1) & 1), abort, p.err);
                tc_fence_after_sync();
                const uint32_t kh = kh0 + buf * TG_OPER;
#pragma unroll
                for (int kk = 0; kk < TG_D / 16; ++kk) {
                    const uint64_t a = umma_sdesc_sw128(kh + (kk >> 2) * TG_TOK * 128 + (kk & 3) * 32, 16, 1024);
                    const uint64_t b = umma_sdesc_sw128(qt + (kk >> 2) * TG_N * 128 + (kk & 3) * 32, 16, 1024);
                    umma_f16_ss(tmem + 16 * buf, a, b, TG_IDESC_S, kk > 0);
                }
                umma_commit(smem_addr(&s_full[buf]));
                umma_commit(smem_addr(&k_free[buf]));
                ++nxt;
                ++c_in;
            };
            bool more = advance();
            if (more) issue_s();
            for (long long ch = 0; more; ++ch) {
                const int buf = int(ch & 1);
                const uint32_t ph = uint32_t((ch >> 1) & 1);
                more = advance();
                // S(ch + 1) of the same segment goes first if its tiles are in by
                // the time P(ch) is; O(ch) never waits for the next chunk's tiles
                const bool early_ok = more && !new_seg;
                bool s_done = false;
                const uint32_t pf = smem_addr(&p_full[buf]);
                const uint32_t cf = smem_addr(&chunk_full[(nxt & 1)]);
                const uint32_t cph = uint32_t((nxt >> 1) & 1);
                const uint64_t t0 = global_timer_ns();
                while (!*abort) {
                    if (early_ok && !s_done && mbar_test(cf, cph)) {
                        issue_s();
                        s_done = true;
                    }
                    if (mbar_test(pf, ph)) break;
                    if (global_timer_ns() - t0 > kWaitLimitNs) {
                        *abort = 1;
                        flag_error(p.err, PKV_DEVERR_TIMEOUT);
                    }
                }
                if (ch >= 2) tg_wait(&o_empty[buf], uint32_t(((ch >> 1) - 1) & 1), abort, p.err);
                tc_fence_after_sync();
                const uint32_t vh = vh0 + buf * TG_OPER, pt = pt0 + buf * TG_QT;
#pragma unroll
                for (int kk = 0; kk < TG_TOK / 16; ++kk) {
                    const uint64_t a = umma_sdesc_sw128(vh + kk * 2048, TG_TOK * 128, 1024);
                    const uint64_t b = umma_sdesc_sw128(pt + (kk >> 2) * TG_N * 128 + (kk & 3) * 32, 16, 1024);
                    umma_f16_ss(tmem + 32 + 16 * buf, a, b, TG_IDESC_O, kk > 0);
                }
                umma_commit(smem_addr(&o_full[buf]));
                umma_commit(smem_addr(&v_free[buf]));
                if (more && !s_done) issue_s();
            }
        }
        __syncwarp();
    } else if (warp >= TG_WG) {
        // ------------------------------------------------------------ dequant warps
        const int slot = warp - TG_WG;
        grid_dep_wait();
        if constexpr (FUSED) fused_write<true, D>(p, warp, TG_COMPUTE_WARPS, tid);
        long long ch = 0;
        Seg sg;
        while (it.next(p, sg)) {
            const int nch = (sg.b1 - sg.b0 + TG_CH - 1) / TG_CH;
            const int new0 = sg.ctx - QL;   // position of the step's first new row
            for (int c = 0; c < nch; ++c, ++ch) {
                const int buf = int(ch & 1);
                const int b = sg.b0 + c * TG_CH + slot;
                const long long j = ch * TG_CH + slot;
                const int st = int(j % S);
                const bool ok = tg_wait(&full[st], uint32_t((j / S) & 1), abort, p.err);
                int ntok = 0;
                if (b < sg.b1 && ok && !poison[st]) ntok = (b == sg.nb - 1) ? sg.ctx - b * kBS : kBS;
                uint8_t* kst = kring + size_t(st) * TG_KST;
                uint8_t* vst = vring + size_t(st) * TG_VST;
                uint8_t* mst = mring + size_t(st) * TG_MST;
                if (FUSED && ntok > 0 && new0 + QL > b * kBS && new0 < (b + 1) * kBS) {
                    // New row jj is "in place" when its slot is that of its own
                    // position: then the tile takes it from k_new / v_new.
                    const size_t tok0 = size_t(sg.s) * QL;
                    const int pos_l = new0 + lane;
                    bool in_place = false;
                    if (lane < QL && tok0 + lane < size_t(p.num_new) && pos_l >= 0 &&
                        pos_l >= visible_lo<false>(p, sg.s, sg.ctx)) {
                        const int64_t my_slot = p.slot_mapping[tok0 + lane];
                        const int my_pb = p.block_tables[size_t(sg.s) * p.max_blocks + pos_l / kBS];
                        in_place = my_slot >= 0 && my_pb >= 0 && my_pb < p.num_blocks &&
                                   my_slot == int64_t(my_pb) * kBS + pos_l % kBS;
                    }
                    const uint32_t mask = __ballot_sync(0xffffffffu, in_place);
                    for (int jj = 0; jj < QL; ++jj) {
                        const int pos = new0 + jj;
                        if (((mask >> jj) & 1u) && pos >= b * kBS && pos < (b + 1) * kBS)
                            tg_patch(kst, vst, mst, pos - b * kBS, tok0 + jj, sg.kvh, lane, p);
                    }
                    __syncwarp();
                }
                // the K tile frees when its score MMA is done; the V tile, the K
                // scales and the mask only when the chunk's O MMA is (the softmax
                // reads the scales and the mask before it lets that MMA go)
                if (ch >= 2) tg_wait(&k_free[buf], uint32_t(((ch >> 1) - 1) & 1), abort, p.err);
                tg_dequant_k(kst, smem + TG_OFF_KH + buf * TG_OPER, slot, ntok, lane);
                if (ch >= 2) tg_wait(&v_free[buf], uint32_t(((ch >> 1) - 1) & 1), abort, p.err);
                tg_dequant_v(vst, mst, smem + TG_OFF_VH + buf * TG_OPER, slot, ntok, lane);
                if (lane < kBS)
                    kscale[buf * TG_TOK + slot * kBS + lane] =
                        lane < ntok ? __half2float(*reinterpret_cast<const __half*>(mst + TG_M_KS + 2 * lane)) : 0.f;
                if (lane == 0) tmask[buf * TG_CH + slot] = ntok > 0 ? (0xffffu >> (kBS - ntok)) : 0u;
                fence_proxy_async_cta();   // the tiles are read by the tensor cores
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&empty[st]);
                    mbar_arrive(&chunk_full[buf]);
                }
            }
        }
    } else {
        // ------------------------------------------------------------ softmax / output warps (0-3)
        constexpr int WT = TG_WG * 32;
        grid_dep_wait();
        // context longer than its table: flagged once per sequence
        for (int s = blockIdx.x * WT + tid; s < p.num_seqs; s += gridDim.x * WT)
            if (p.context_lens[s] > p.max_blocks * kBS) flag_error(p.err, PKV_DEVERR_CAPACITY);
        if constexpr (FUSED) fused_write<true, D>(p, warp, TG_COMPUTE_WARPS, tid);
        // sequences with nothing visible still get their zero rows
        for (int s = blockIdx.x; s < p.num_seqs; s += gridDim.x)
            if (seq_ctx(p, s) == 0)
                for (int i = tid; i < QL * H * D; i += WT) store_out(p.out, p.out_dtype, size_t(s) * QL * H * D + i, 0.f);
        // P rows of padding columns: zero once (their products are never read)
        for (int i = tid; i < 2 * TG_QT / 16; i += WT)
            *reinterpret_cast<uint4*>(smem + TG_OFF_P + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
        const int t = tid;                 // token row of a chunk / head-dim row of O^T
        const int dim = tg_dim_of(t);
        const uint32_t tl = uint32_t(32 * warp) << 16;   // this warp's tensor-memory lanes
        const uint32_t qt = smem_addr(smem + TG_OFF_Q);
        long long ch = 0;
        Seg sg;
        while (it.next(p, sg)) {
            const int nch = (sg.b1 - sg.b0 + TG_CH - 1) / TG_CH;
            if (nch == 0) continue;
            const int lo = visible_lo<false>(p, sg.s, sg.ctx);
            // ---- the segment's query tile: rows n < MQ (head n / q_len, draft n % q_len), zero below
            for (int e = t; e < TG_N * (D / 8); e += WT) {
                const int n = e / (D / 8), d0 = 8 * (e % (D / 8));
                uint32_t hw[4] = {0u, 0u, 0u, 0u};
                if (n < MQ) {
                    const size_t qoff = ((size_t(sg.s) * QL + n % QL) * H + sg.kvh * G + n / QL) * D + d0;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        hw[i] = pack2<false>(load_q(p.q, p.q_dtype, qoff + 2 * i), load_q(p.q, p.q_dtype, qoff + 2 * i + 1));
                }
                sts_u32(qt + sw128_off(n, d0, TG_N), hw[0]);
                sts_u32(qt + sw128_off(n, d0, TG_N) + 4, hw[1]);
                sts_u32(qt + sw128_off(n, d0, TG_N) + 8, hw[2]);
                sts_u32(qt + sw128_off(n, d0, TG_N) + 12, hw[3]);
            }
            fence_proxy_async_cta();
            named_barrier_sync(1, WT);
            if (t == 0) mbar_arrive(q_ready);
            float o_run[NV], l_part[NV], m_run[NV], a_prev[NV];
            int lim[NV];
#pragma unroll
            for (int n = 0; n < NV; ++n) {
                o_run[n] = 0.f;
                l_part[n] = 0.f;
                m_run[n] = -INFINITY;
                a_prev[n] = 1.f;
                lim[n] = n < MQ ? max(0, sg.ctx - QL + (n % QL) + 1) : 0;   // draft j sees ctx - q_len + j + 1 tokens
            }
            auto fold = [&](long long k) {   // O^T of chunk k into the running output
                const int fb = int(k & 1);
                tg_wait(&o_full[fb], uint32_t((k >> 1) & 1), abort, p.err);
                tc_fence_after_sync();
                float ov[16];
                tmem_ld16(tmem + tl + 32 + 16 * fb, ov);
#pragma unroll
                for (int n = 0; n < NV; ++n) o_run[n] = fmaf(o_run[n], a_prev[n], ov[n]);
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&o_empty[fb]);
            };
            for (int c = 0; c < nch; ++c, ++ch) {
                const int buf = int(ch & 1);
                tg_wait(&s_full[buf], uint32_t((ch >> 1) & 1), abort, p.err);
                tc_fence_after_sync();
                float sv[16];
                tmem_ld16(tmem + tl + 16 * buf, sv);
                const int pos = (sg.b0 + c * TG_CH) * kBS + t;
                const bool valid = ((tmask[buf * TG_CH + (t >> 4)] >> (t & 15)) & 1u) && pos >= lo;
                const float kq = kscale[buf * TG_TOK + t] * p.scale_log2;
                float x[NV];
#pragma unroll
                for (int n = 0; n < NV; ++n) {
                    x[n] = (valid && pos < lim[n]) ? sv[n] * kq : -INFINITY;
                    float m = x[n];
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                    if (lane == 0) colx[(buf * TG_WG + warp) * TG_N + n] = m;
                }
                // one barrier per chunk: the column maxima are double-buffered, and a
                // warp can rewrite buffer b only after every warp has passed the
                // next chunk's barrier, i.e. has read b
                named_barrier_sync(1, WT);
                float alpha[NV];
#pragma unroll
                for (int n = 0; n < NV; ++n) {
                    float cm = colx[buf * TG_WG * TG_N + n];
#pragma unroll
                    for (int w2 = 1; w2 < TG_WG; ++w2) cm = fmaxf(cm, colx[(buf * TG_WG + w2) * TG_N + n]);
                    const float mn = fmaxf(m_run[n], cm);
                    const float mu = (mn == -INFINITY) ? 0.f : mn;
                    alpha[n] = exp2f(m_run[n] - mu);
                    const float pn = exp2f(x[n] - mu);
                    l_part[n] = fmaf(l_part[n], alpha[n], pn);
                    m_run[n] = mn;
                    if (n < MQ) {
                        const __half hp = __float2half_rn(pn);
                        sts_u16(smem_addr(smem + TG_OFF_P + buf * TG_QT) + sw128_off(n, t, TG_N), __half_as_ushort(hp));
                    }
                }
                fence_proxy_async_cta();   // P is read by the tensor cores
                tc_fence_before_sync();    // this warp's scores are read: S(buf) may be rewritten
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[buf]);
                if (c > 0) fold(ch - 1);
#pragma unroll
                for (int n = 0; n < NV; ++n) a_prev[n] = alpha[n];
            }
            fold(ch - 1);
            // ---- the segment's row sums, then its output or its piece
#pragma unroll
            for (int n = 0; n < NV; ++n) {
                float l = l_part[n];
#pragma unroll
                for (int o = 16; o >= 1; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
                if (lane == 0) lsum[warp * TG_N + n] = l;
            }
            named_barrier_sync(1, WT);
            float L[NV];
#pragma unroll
            for (int n = 0; n < NV; ++n) {
                L[n] = lsum[n];
#pragma unroll
                for (int w2 = 1; w2 < TG_WG; ++w2) L[n] += lsum[w2 * TG_N + n];
            }
            const int pair = sg.s * Hkv + sg.kvh;
            const bool piece = !sg.whole;
            if (!piece) {
#pragma unroll
                for (int n = 0; n < NV; ++n) {
                    if (n >= MQ) break;
                    const bool live = L[n] > 0.f;
                    const size_t row = size_t(sg.s) * QL + n % QL;
                    store_out(p.out, p.out_dtype, (row * H + sg.kvh * G + n / QL) * D + dim, live ? o_run[n] / L[n] : 0.f);
                }
            } else {
                // unnormalised piece partial into the workspace slot (lane_idx + s) * Hkv + kvh
                const int slot = (lane_idx + sg.s) * Hkv + sg.kvh;
#pragma unroll
                for (int n = 0; n < NV; ++n) {
                    if (n >= MQ) break;
                    p.part_o[(size_t(slot) * kMaxRows + n) * D + dim] = o_run[n];
                    if (t == 0)
                        reinterpret_cast<float2*>(p.part_ml)[size_t(slot) * kMaxRows + n] = make_float2(m_run[n], L[n]);
                }
                named_barrier_sync(1, WT);
                const int c_lo = int((sg.pair_start + sg.cost_base - p.seg_cost) / chunk),
                          c_hi = int((sg.pair_start + sg.nu - 1 + sg.cost_base - p.seg_cost) / chunk);
                const int np = c_hi - c_lo + 1;
                if (t == 0) {
                    __threadfence();
                    const int prev = atomicAdd(&p.counters[pair], 1);
                    __threadfence();   // acquire: the other pieces' partials before our loads
                    flag[1] = (prev == np - 1) ? 1 : 0;
                }
                named_barrier_sync(1, WT);
                if (flag[1]) {
                    // the last piece combines all of them in piece order (own piece from registers)
                    const int own = lane_idx - c_lo;
#pragma unroll
                    for (int n = 0; n < NV; ++n) {
                        if (n >= MQ) break;
                        float acc = 0.f, Mr = -INFINITY, Lr = 0.f;
                        for (int c0 = 0; c0 < np; c0 += 8) {
                            float2 ml[8];
                            float v[8];
#pragma unroll
                            for (int u = 0; u < 8; ++u) {
                                const int cc = c0 + u;
                                ml[u] = make_float2(-INFINITY, 0.f);
                                v[u] = 0.f;
                                if (cc == own) {
                                    ml[u] = make_float2(m_run[n], L[n]);
                                    v[u] = o_run[n];
                                } else if (cc < np) {
                                    const size_t sl = size_t((c_lo + cc + sg.s) * Hkv + sg.kvh) * kMaxRows + n;
                                    ml[u] = __ldcg(reinterpret_cast<const float2*>(p.part_ml) + sl);
                                    v[u] = __ldcg(p.part_o + sl * D + dim);
                                }
                            }
                            float Mn = Mr;
#pragma unroll
                            for (int u = 0; u < 8; ++u)
                                if (ml[u].y > 0.f) Mn = fmaxf(Mn, ml[u].x);
                            const float a = (Mr == -INFINITY) ? 0.f : exp2f(Mr - Mn);
                            acc *= a;
                            Lr *= a;
#pragma unroll
                            for (int u = 0; u < 8; ++u) {
                                const float f = (ml[u].y > 0.f) ? exp2f(ml[u].x - Mn) : 0.f;
                                acc = fmaf(f, v[u], acc);
                                Lr = fmaf(f, ml[u].y, Lr);
                            }
                            Mr = Mn;
                        }
                        const size_t row = size_t(sg.s) * QL + n % QL;
                        store_out(p.out, p.out_dtype, (row * H + sg.kvh * G + n / QL) * D + dim, Lr > 0.f ? acc / Lr : 0.f);
                    }
                    if (t == 0) p.counters[pair] = 0;   // ready for the next launch
                }
            }
            named_barrier_sync(1, WT);   // lsum / colx / flag reused by the next segment
        }
    }

    // ---- every warp: tensor memory back before the CTA exits
    tc_fence_before_sync();
    __syncthreads();
    if (warp == TG_MMA_WARP) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TG_TMEM_COLS);
    }
}

template <int NV, bool FUSED>
cudaError_t launch_tg(AttnParams p, const CUtensorMap& km, const CUtensorMap& vm, cudaStream_t stream) {
    static int num_sms = 0;
    if (num_sms == 0) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    int stages = 0;
    while (tg_smem_bytes(stages + TG_CH) <= kSmemLimit) stages += TG_CH;
    if (stages < TG_CH) return cudaErrorInvalidConfiguration;
    p.stages = stages;
    static bool attr_set = false;
    if (!attr_set) {
        cudaError_t e = cudaFuncSetAttribute(attention_tg_kernel<NV, FUSED>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemLimit);
        if (e != cudaSuccess) return e;
        attr_set = true;
    }
    const int cap = num_sms < kMaxGrid ? num_sms : kMaxGrid;
    int L = cap / p.num_kv_heads;
    if (L < 1) L = 1;
    const long long lane_units = (long long)p.num_seqs * p.max_blocks;
    if (lane_units < L) L = int(lane_units < 1 ? 1 : lane_units);
    return launch_kernel(attention_tg_kernel<NV, FUSED>, dim3(L * p.num_kv_heads), dim3(TG_THREADS),
                         size_t(tg_smem_bytes(stages)), stream, km, vm, p);
}

}  // namespace

// Not dispatched: at every shape measured (K8/V4 batch 32, 4 to 16 query rows
// per kv head) the mma.sync math of attention_impl.cuh is faster.
bool attention_tg_supported(int, int, int, int, int) { return false; }

cudaError_t launch_attention_tg(const AttnParams& p, int gqa, const CUtensorMap& km, const CUtensorMap& vm,
                                cudaStream_t stream) {
    const int mq = gqa * p.q_len;
    const bool fused = p.num_new > 0;
    if (mq <= 4) return fused ? launch_tg<4, true>(p, km, vm, stream) : launch_tg<4, false>(p, km, vm, stream);
    if (mq <= 8) return fused ? launch_tg<8, true>(p, km, vm, stream) : launch_tg<8, false>(p, km, vm, stream);
    return fused ? launch_tg<16, true>(p, km, vm, stream) : launch_tg<16, false>(p, km, vm, stream);
}

}  // namespace pkv
