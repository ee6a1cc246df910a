// api.cu -- the extern "C" boundary declared in include/pkv.h: host-side
// argument checks, TMA tensor-map encoding and kernel dispatch.  Nothing here
// allocates device memory and nothing is cached between calls.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <string>

#include "pkv.h"
#include "pkv_internal.h"

namespace pkv {

bool pdl_enabled() {
    static const bool on = [] {
        const char* v = std::getenv("PKV_PDL");
        return !(v && v[0] == '0' && v[1] == '\0');
    }();
    return on;
}

}  // namespace pkv

namespace {

thread_local std::string g_last_error;

pkv_status fail(pkv_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

pkv_status ok() {
    g_last_error.clear();
    return PKV_OK;
}

pkv_status cuda_result(cudaError_t e, const char* what) {
    if (e == cudaSuccess) return ok();
    return fail(PKV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

#define CHECK_PTR(ptr, name)                                                                          \
    do {                                                                                              \
        if ((ptr) == nullptr) return fail(PKV_ERR_INVALID_ARG, "%s is NULL", name);                   \
        if (!aligned16(ptr)) return fail(PKV_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);     \
    } while (0)

pkv_status check_cache(const pkv_cache* c, bool need_half) {
    if (!c) return fail(PKV_ERR_INVALID_ARG, "cache is NULL");
    if (c->kind != PKV_CACHE_F16 && c->kind != PKV_CACHE_BF16 && c->kind != PKV_CACHE_K8V4)
        return fail(PKV_ERR_INVALID_ARG, "unknown cache kind %d", c->kind);
    if (need_half && c->kind == PKV_CACHE_K8V4)
        return fail(PKV_ERR_INVALID_ARG, "this call needs an fp16 or bf16 cache");
    if (c->block_size != 16) return fail(PKV_ERR_UNSUPPORTED, "block_size %d (only 16)", c->block_size);
    if (c->head_dim != 64 && c->head_dim != 128)
        return fail(PKV_ERR_UNSUPPORTED, "head_dim %d (64 or 128)", c->head_dim);
    if (c->num_kv_heads < 1 || c->num_kv_heads > 65535)
        return fail(PKV_ERR_INVALID_ARG, "num_kv_heads %d", c->num_kv_heads);
    if (c->num_blocks < 1 || int64_t(c->num_blocks) * 16 > INT32_MAX)
        return fail(PKV_ERR_INVALID_ARG, "num_blocks %d", c->num_blocks);
    CHECK_PTR(c->k, "cache->k");
    CHECK_PTR(c->v, "cache->v");
    if (c->kind == PKV_CACHE_K8V4) {
        if (c->v_group != 32) return fail(PKV_ERR_UNSUPPORTED, "v_group %d (only 32)", c->v_group);
        CHECK_PTR(c->k_scale, "cache->k_scale");
        CHECK_PTR(c->v_scale, "cache->v_scale");
        CHECK_PTR(c->v_zero, "cache->v_zero");
    }
    return PKV_OK;
}

pkv_status check_seqs(const pkv_seqs* s) {
    if (!s) return fail(PKV_ERR_INVALID_ARG, "seqs is NULL");
    if (s->num_seqs < 0 || s->num_seqs > 65535) return fail(PKV_ERR_INVALID_ARG, "num_seqs %d", s->num_seqs);
    if (s->q_len < 1) return fail(PKV_ERR_INVALID_ARG, "q_len %d", s->q_len);
    if (s->sliding_window < 0) return fail(PKV_ERR_INVALID_ARG, "sliding_window %d", s->sliding_window);
    if (s->max_blocks_per_seq < 1) return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq %d", s->max_blocks_per_seq);
    if (int64_t(s->max_blocks_per_seq) * 16 > INT32_MAX / 2)
        return fail(PKV_ERR_INVALID_ARG, "max_blocks_per_seq %d too large", s->max_blocks_per_seq);
    if (s->num_seqs > 0) {
        if (!s->block_tables) return fail(PKV_ERR_INVALID_ARG, "seqs->block_tables is NULL");
        if (!s->context_lens) return fail(PKV_ERR_INVALID_ARG, "seqs->context_lens is NULL");
    }
    return PKV_OK;
}

int cache_dtype(const pkv_cache* c) { return c->kind == PKV_CACHE_BF16 ? PKV_BF16 : PKV_F16; }

// ---------------------------------------------------------------- tensor maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// A 2-D view of a paged cache tensor: rows = num_blocks*16 token slots, each
// row `row_bytes` long; box = one kv head's `box_bytes` of 16 consecutive rows.
pkv_status tile_map(CUtensorMap* map, void* base, int64_t rows, int64_t row_bytes, int box_bytes,
                    CUtensorMapSwizzle swz) {
    auto fn = encode_fn();
    if (!fn) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    cuuint64_t dims[2] = {cuuint64_t(row_bytes), cuuint64_t(rows)};
    cuuint64_t strides[1] = {cuuint64_t(row_bytes)};
    cuuint32_t box[2] = {cuuint32_t(box_bytes), 16u};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
    return PKV_OK;
}

// A 3-D view for the tensor-core tiles of fp16/bf16 caches: {128-byte chunk,
// token slot, chunk index across the row}.  One box {128, 16, D/64} is a kv
// head's 16 rows, landing chunk-major as D/64 sub-tiles of 16 x 128 bytes (the
// layout the 128B swizzle and ldmatrix want), in a single copy operation.
pkv_status chunk_map(CUtensorMap* map, void* base, int64_t rows, int64_t row_bytes, int head_dim) {
    auto fn = encode_fn();
    if (!fn) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable from the driver");
    cuuint64_t dims[3] = {128u, cuuint64_t(rows), cuuint64_t(row_bytes / 128)};
    cuuint64_t strides[2] = {cuuint64_t(row_bytes), 128u};
    cuuint32_t box[3] = {128u, 16u, cuuint32_t(head_dim / 64)};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, base, dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(PKV_ERR_CUDA, "cuTensorMapEncodeTiled (3-D) failed (%d)", int(r));
    return PKV_OK;
}

CUtensorMapSwizzle swizzle_for(int row_bytes) {
    return row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                            : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
}

// CUDA-core kernel: one box per tile (16 rows x one kv head), no swizzle.
// Tensor-core kernel: swizzled rows of at most 128 bytes, so that the ldmatrix /
// 128-bit reads of a tile are conflict-free (fp16/bf16: 64-dim chunks with the
// 128B swizzle, one 3-D box; K8: the whole D-byte row; V4: the whole D/2-byte row).
pkv_status cache_maps(const pkv_cache* c, CUtensorMap* km, CUtensorMap* vm, bool tc) {
    const int64_t rows = int64_t(c->num_blocks) * 16;
    const int D = c->head_dim, H = c->num_kv_heads;
    pkv_status st;
    if (c->kind == PKV_CACHE_K8V4) {
        st = tile_map(km, c->k, rows, int64_t(H) * D, D, swizzle_for(D));
        if (st != PKV_OK) return st;
        return tile_map(vm, c->v, rows, int64_t(H) * D / 2, D / 2, swizzle_for(D / 2));
    }
    if (tc) {
        st = chunk_map(km, c->k, rows, int64_t(H) * D * 2, D);
        if (st != PKV_OK) return st;
        return chunk_map(vm, c->v, rows, int64_t(H) * D * 2, D);
    }
    st = tile_map(km, c->k, rows, int64_t(H) * D * 2, D * 2, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (st != PKV_OK) return st;
    return tile_map(vm, c->v, rows, int64_t(H) * D * 2, D * 2, CU_TENSOR_MAP_SWIZZLE_NONE);
}

#ifdef PKV_TIMELINE
// Timeline build only: the device buffer the attention kernels stamp (see
// attention_impl.cuh); set by pkv_timeline_attach, read by every later call.
unsigned long long* g_timeline = nullptr;
#endif

// Shared checks + parameter block of both attention entry points.
pkv_status attn_setup(pkv::AttnParams* p, const void* q, pkv_dtype q_dtype, int32_t num_heads, float scale,
                      const pkv_cache* cache, const pkv_seqs* seqs, uint32_t* err, int* gqa) {
    pkv_status st = check_cache(cache, false);
    if (st != PKV_OK) return st;
    if ((st = check_seqs(seqs)) != PKV_OK) return st;
    CHECK_PTR(q, "q");
    if (q_dtype != PKV_F16 && q_dtype != PKV_BF16) return fail(PKV_ERR_INVALID_ARG, "q_dtype %d", q_dtype);
    if (cache->kind != PKV_CACHE_K8V4 && q_dtype != cache_dtype(cache))
        return fail(PKV_ERR_INVALID_ARG, "q_dtype must match the fp16/bf16 cache dtype");
    if (num_heads < 1 || num_heads % cache->num_kv_heads != 0)
        return fail(PKV_ERR_INVALID_ARG, "num_heads %d is not a multiple of num_kv_heads %d", num_heads,
                    cache->num_kv_heads);
    *gqa = num_heads / cache->num_kv_heads;
    if (*gqa != 1 && *gqa != 2 && *gqa != 4 && *gqa != 8)
        return fail(PKV_ERR_UNSUPPORTED, "group size %d (1, 2, 4 or 8)", *gqa);
    if (!(scale == scale)) return fail(PKV_ERR_INVALID_ARG, "scale is NaN");
    if (!pkv::attention_supported(cache->kind, cache->head_dim, *gqa, seqs->q_len))
        return fail(PKV_ERR_UNSUPPORTED, "no kernel for cache kind %d, head_dim %d, group %d, q_len %d", cache->kind,
                    cache->head_dim, *gqa, seqs->q_len);
    *p = pkv::AttnParams{};
#ifdef PKV_TIMELINE
    p->timeline = g_timeline;
#endif
    p->q = q;
    p->q_dtype = q_dtype;
    p->scale_log2 = scale * 1.4426950408889634f;
    p->num_heads = num_heads;
    p->num_kv_heads = cache->num_kv_heads;
    p->q_len = seqs->q_len;
    p->num_blocks = cache->num_blocks;
    p->head_dim = cache->head_dim;
    p->k_scale = cache->k_scale;
    p->v_scale = cache->v_scale;
    p->v_zero = cache->v_zero;
    p->block_tables = seqs->block_tables;
    p->context_lens = seqs->context_lens;
    p->num_seqs = seqs->num_seqs;
    p->max_blocks = seqs->max_blocks_per_seq;
    p->window = seqs->sliding_window;
    p->err = err;
    return PKV_OK;
}

pkv_status attn_launch(pkv::AttnParams p, const pkv_cache* cache, int gqa, pkv_stream_t stream) {
    const bool tc = pkv::attention_uses_tensor_cores(cache->kind, p.q_len, gqa, pkv::is_cascade_pass(p));
    CUtensorMap km, vm;
    pkv_status st = cache_maps(cache, &km, &vm, tc);
    if (st != PKV_OK) return st;
    return cuda_result(pkv::launch_attention(p, cache->kind, gqa, km, vm, reinterpret_cast<cudaStream_t>(stream)),
                       "attention launch");
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

#ifdef PKV_TIMELINE
extern "C" void pkv_timeline_attach(void* device_buffer) {
    g_timeline = static_cast<unsigned long long*>(device_buffer);
}
#endif

extern "C" {

pkv_status pkv_reshape_and_cache(const pkv_cache* cache, const void* k_new, const void* v_new,
                                 const int64_t* slot_mapping, int32_t num_tokens, uint32_t* err_flags,
                                 pkv_stream_t stream) {
    pkv_status st = check_cache(cache, true);
    if (st != PKV_OK) return st;
    if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_tokens %d", num_tokens);
    if (num_tokens == 0) return ok();
    CHECK_PTR(k_new, "k_new");
    CHECK_PTR(v_new, "v_new");
    if (!slot_mapping) return fail(PKV_ERR_INVALID_ARG, "slot_mapping is NULL");
    pkv::CacheWriteParams p{};
    p.k_cache = cache->k;
    p.v_cache = cache->v;
    p.k_new = k_new;
    p.v_new = v_new;
    p.slot_mapping = slot_mapping;
    p.num_tokens = num_tokens;
    p.num_blocks = cache->num_blocks;
    p.num_kv_heads = cache->num_kv_heads;
    p.head_dim = cache->head_dim;
    p.err = err_flags;
    return cuda_result(pkv::launch_reshape_and_cache(p, 2, reinterpret_cast<cudaStream_t>(stream)),
                       "reshape_and_cache launch");
}

pkv_status pkv_quantize_kv(const pkv_cache* cache, const void* k_new, const void* v_new, pkv_dtype src_dtype,
                           const int64_t* slot_mapping, int32_t num_tokens, uint32_t* err_flags,
                           pkv_stream_t stream) {
    pkv_status st = check_cache(cache, false);
    if (st != PKV_OK) return st;
    if (cache->kind != PKV_CACHE_K8V4) return fail(PKV_ERR_INVALID_ARG, "quantize_kv needs a K8V4 cache");
    if (src_dtype != PKV_F16 && src_dtype != PKV_BF16) return fail(PKV_ERR_INVALID_ARG, "src_dtype %d", src_dtype);
    if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_tokens %d", num_tokens);
    if (num_tokens == 0) return ok();
    CHECK_PTR(k_new, "k_new");
    CHECK_PTR(v_new, "v_new");
    if (!slot_mapping) return fail(PKV_ERR_INVALID_ARG, "slot_mapping is NULL");
    pkv::CacheWriteParams p{};
    p.k_cache = cache->k;
    p.v_cache = cache->v;
    p.k_new = k_new;
    p.v_new = v_new;
    p.slot_mapping = slot_mapping;
    p.num_tokens = num_tokens;
    p.num_blocks = cache->num_blocks;
    p.num_kv_heads = cache->num_kv_heads;
    p.head_dim = cache->head_dim;
    p.err = err_flags;
    p.k_scale = cache->k_scale;
    p.v_scale = cache->v_scale;
    p.v_zero = cache->v_zero;
    p.src_dtype = src_dtype;
    return cuda_result(pkv::launch_quantize_kv(p, reinterpret_cast<cudaStream_t>(stream)), "quantize_kv launch");
}

pkv_status pkv_paged_attention(void* out, pkv_dtype out_dtype, const void* q, pkv_dtype q_dtype, int32_t num_heads,
                               float scale, const pkv_cache* cache, const pkv_seqs* seqs, uint32_t* err_flags,
                               pkv_stream_t stream) {
    pkv::AttnParams p;
    int gqa = 0;
    pkv_status st = attn_setup(&p, q, q_dtype, num_heads, scale, cache, seqs, err_flags, &gqa);
    if (st != PKV_OK) return st;
    CHECK_PTR(out, "out");
    if (out_dtype != PKV_F16 && out_dtype != PKV_BF16 && out_dtype != PKV_F32)
        return fail(PKV_ERR_INVALID_ARG, "out_dtype %d", out_dtype);
    if (seqs->num_seqs == 0) return ok();
    p.out = out;
    p.out_dtype = out_dtype;
    p.partition_blocks = seqs->max_blocks_per_seq;
    p.max_partitions = 1;
    p.mode = pkv::kModeSingle;
    return attn_launch(p, cache, gqa, stream);
}

size_t pkv_split_workspace_bytes(int32_t num_rows, int32_t num_heads, int32_t head_dim, int32_t max_partitions) {
    if (num_rows <= 0 || num_heads <= 0 || head_dim <= 0 || max_partitions <= 0) return 0;
    const size_t n = size_t(num_rows) * size_t(num_heads) * size_t(max_partitions);
    return align256(n * size_t(head_dim) * 4) + 2 * align256(n * 4);
}

pkv_status pkv_paged_attention_split(float* tmp_out, float* max_logits, float* exp_sums, int32_t partition_size,
                                     int32_t max_partitions, const void* q, pkv_dtype q_dtype, int32_t num_heads,
                                     float scale, const pkv_cache* cache, const pkv_seqs* seqs,
                                     uint32_t* err_flags, pkv_stream_t stream) {
    pkv::AttnParams p;
    int gqa = 0;
    pkv_status st = attn_setup(&p, q, q_dtype, num_heads, scale, cache, seqs, err_flags, &gqa);
    if (st != PKV_OK) return st;
    CHECK_PTR(tmp_out, "tmp_out");
    CHECK_PTR(max_logits, "max_logits");
    CHECK_PTR(exp_sums, "exp_sums");
    if (partition_size < 16 || partition_size % 16 != 0)
        return fail(PKV_ERR_INVALID_ARG, "partition_size %d is not a positive multiple of 16", partition_size);
    if (max_partitions < 1 || max_partitions > 65535)
        return fail(PKV_ERR_INVALID_ARG, "max_partitions %d", max_partitions);
    if (int64_t(max_partitions) * partition_size < int64_t(seqs->max_blocks_per_seq) * 16)
        return fail(PKV_ERR_INVALID_ARG, "max_partitions * partition_size (%lld) does not cover the block table (%lld)",
                    (long long)max_partitions * partition_size, (long long)seqs->max_blocks_per_seq * 16);
    if (seqs->num_seqs == 0) return ok();
    p.tmp_out = tmp_out;
    p.max_logits = max_logits;
    p.exp_sums = exp_sums;
    p.partition_blocks = partition_size / 16;
    p.max_partitions = max_partitions;
    p.mode = pkv::kModeSplit;
    return attn_launch(p, cache, gqa, stream);
}

size_t pkv_balanced_workspace_bytes(int32_t num_seqs, int32_t num_kv_heads, int32_t head_dim) {
    if (num_seqs <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
    return pkv::balanced_workspace_bytes(num_seqs, num_kv_heads, head_dim);
}

}  // extern "C"

namespace {

// Output, workspace and schedule of the balanced entry points (after attn_setup).
pkv_status balanced_setup(pkv::AttnParams& p, void* out, pkv_dtype out_dtype, const pkv_cache* cache,
                          const pkv_seqs* seqs, void* workspace, size_t workspace_bytes) {
    CHECK_PTR(out, "out");
    if (out_dtype != PKV_F16 && out_dtype != PKV_BF16 && out_dtype != PKV_F32)
        return fail(PKV_ERR_INVALID_ARG, "out_dtype %d", out_dtype);
    if (cache->num_kv_heads > pkv::kMaxGrid)
        return fail(PKV_ERR_UNSUPPORTED, "num_kv_heads %d above %d for the balanced schedule", cache->num_kv_heads,
                    pkv::kMaxGrid);
    if (seqs->num_seqs == 0) return ok();
    const size_t need = pkv::balanced_workspace_bytes(seqs->num_seqs, cache->num_kv_heads, cache->head_dim);
    if (!workspace) return fail(PKV_ERR_INVALID_ARG, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(PKV_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
    if (workspace_bytes < need)
        return fail(PKV_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
    const size_t pairs = size_t(seqs->num_seqs) * size_t(cache->num_kv_heads);
    const size_t slots = size_t(pkv::kMaxGrid) + pairs;
    uint8_t* w = static_cast<uint8_t*>(workspace);
    p.part_o = reinterpret_cast<float*>(w);
    w += align256(slots * 16 * size_t(cache->head_dim) * 4);
    p.part_ml = reinterpret_cast<float*>(w);
    w += align256(slots * 16 * 2 * 4);
    p.counters = reinterpret_cast<int32_t*>(w);
    p.out = out;
    p.out_dtype = out_dtype;
    p.partition_blocks = seqs->max_blocks_per_seq;
    p.max_partitions = 1;
    p.mode = pkv::kModeBalanced;
    p.min_chunk = pkv::kMinChunk;
    p.seg_cost = pkv::kSegCost;
    return ok();
}

}  // namespace

extern "C" {

pkv_status pkv_paged_attention_balanced(void* out, pkv_dtype out_dtype, const void* q, pkv_dtype q_dtype,
                                        int32_t num_heads, float scale, const pkv_cache* cache, const pkv_seqs* seqs,
                                        void* workspace, size_t workspace_bytes, uint32_t* err_flags,
                                        pkv_stream_t stream) {
    pkv::AttnParams p;
    int gqa = 0;
    pkv_status st = attn_setup(&p, q, q_dtype, num_heads, scale, cache, seqs, err_flags, &gqa);
    if (st != PKV_OK) return st;
    if ((st = balanced_setup(p, out, out_dtype, cache, seqs, workspace, workspace_bytes)) != PKV_OK) return st;
    if (seqs->num_seqs == 0) return ok();
    return attn_launch(p, cache, gqa, stream);
}

size_t pkv_cascade_workspace_bytes(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                   int32_t num_items, int32_t item_width) {
    if (num_seqs < 0 || num_heads < 1 || num_kv_heads < 1 || head_dim < 1 || num_items < 0 || item_width < 1 ||
        item_width > 16)
        return 0;
    const size_t rh2 = size_t(num_seqs) * size_t(num_heads) * 2;
    const size_t list = size_t(num_items) + size_t(num_seqs);
    return align256(rh2 * size_t(head_dim) * 4) + 2 * align256(rh2 * 4) + 3 * align256(list * 4) +
           align256(list * size_t(item_width) * 4) + pkv::balanced_workspace_bytes(int(list), num_kv_heads, head_dim);
}

pkv_status pkv_paged_attention_cascade(void* out, pkv_dtype out_dtype, const void* q, pkv_dtype q_dtype,
                                       int32_t num_heads, float scale, const pkv_cache* cache, const pkv_seqs* seqs,
                                       const int32_t* members, const int32_t* item_blocks, int32_t num_items,
                                       int32_t item_width, void* workspace, size_t workspace_bytes,
                                       uint32_t* err_flags, pkv_stream_t stream) {
    pkv::AttnParams p;
    int gqa = 0;
    pkv_status st = attn_setup(&p, q, q_dtype, num_heads, scale, cache, seqs, err_flags, &gqa);
    if (st != PKV_OK) return st;
    if (seqs->q_len != 1) return fail(PKV_ERR_UNSUPPORTED, "cascade attention is for q_len 1 decode");
    if (seqs->sliding_window != 0) return fail(PKV_ERR_UNSUPPORTED, "cascade attention with a sliding window");
    if (num_items < 0) return fail(PKV_ERR_INVALID_ARG, "num_items %d", num_items);
    if (item_width < 1 || gqa * item_width > 16)
        return fail(PKV_ERR_UNSUPPORTED, "item_width %d: group size x item width must be 1..16", item_width);
    if (num_items > 0 && (!members || !item_blocks)) return fail(PKV_ERR_INVALID_ARG, "members / item_blocks is NULL");
    if ((int64_t(num_items) + seqs->num_seqs) * item_width > INT32_MAX / 2 ||
        (int64_t(num_items) + seqs->num_seqs) * cache->num_kv_heads > INT32_MAX / 2)
        return fail(PKV_ERR_INVALID_ARG, "too many items");
    if (!pkv::attention_supported(cache->kind, cache->head_dim, gqa, item_width < 2 ? 2 : item_width))
        return fail(PKV_ERR_UNSUPPORTED, "no cascade kernel for this shape");
    if (cache->num_kv_heads > pkv::kMaxGrid)
        return fail(PKV_ERR_UNSUPPORTED, "num_kv_heads %d above %d", cache->num_kv_heads, pkv::kMaxGrid);
    CHECK_PTR(out, "out");
    if (out_dtype != PKV_F16 && out_dtype != PKV_BF16 && out_dtype != PKV_F32)
        return fail(PKV_ERR_INVALID_ARG, "out_dtype %d", out_dtype);
    if (seqs->num_seqs == 0) return ok();
    const size_t need = pkv_cascade_workspace_bytes(seqs->num_seqs, num_heads, cache->num_kv_heads, cache->head_dim,
                                                    num_items, item_width);
    if (!workspace) return fail(PKV_ERR_INVALID_ARG, "workspace is NULL");
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return fail(PKV_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
    if (workspace_bytes < need)
        return fail(PKV_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
    const size_t rh2 = size_t(seqs->num_seqs) * size_t(num_heads) * 2;
    const size_t list = size_t(num_items) + size_t(seqs->num_seqs);
    const size_t pairs = list * size_t(cache->num_kv_heads);
    const size_t piece_slots = size_t(pkv::kMaxGrid) + pairs;
    uint8_t* w = static_cast<uint8_t*>(workspace);
    float* tmp_out = reinterpret_cast<float*>(w);
    w += align256(rh2 * size_t(cache->head_dim) * 4);
    float* max_logits = reinterpret_cast<float*>(w);
    w += align256(rh2 * 4);
    float* exp_sums = reinterpret_cast<float*>(w);
    w += align256(rh2 * 4);
    int32_t* list_ctx = reinterpret_cast<int32_t*>(w);
    w += align256(list * 4);
    int32_t* list_seq = reinterpret_cast<int32_t*>(w);
    w += align256(list * 4);
    int32_t* list_start = reinterpret_cast<int32_t*>(w);
    w += align256(list * 4);
    int32_t* list_rows = reinterpret_cast<int32_t*>(w);
    w += align256(list * size_t(item_width) * 4);
    p.part_o = reinterpret_cast<float*>(w);
    w += align256(piece_slots * 16 * size_t(cache->head_dim) * 4);
    p.part_ml = reinterpret_cast<float*>(w);
    w += align256(piece_slots * 16 * 2 * 4);
    p.counters = reinterpret_cast<int32_t*>(w);
    cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);

    pkv::CascadeParams c{};
    c.members = members;
    c.item_blocks = item_blocks;
    c.block_tables = seqs->block_tables;
    c.context_lens = seqs->context_lens;
    c.num_items = num_items;
    c.width = item_width;
    c.num_seqs = seqs->num_seqs;
    c.max_blocks = seqs->max_blocks_per_seq;
    c.list_ctx = list_ctx;
    c.list_seq = list_seq;
    c.list_start = list_start;
    c.list_rows = list_rows;
    c.counters = p.counters;
    c.num_counters = int32_t(pairs);
    c.err = err_flags;
    cudaError_t e = pkv::launch_cascade_setup(c, cs);
    if (e != cudaSuccess) return cuda_result(e, "cascade set-up launch");
    // one balanced pass over the list: an item's combined partial goes to slot 1
    // of its members' rows, a sequence's own to slot 0
    p.tmp_out = tmp_out;
    p.max_logits = max_logits;
    p.exp_sums = exp_sums;
    p.partition_blocks = seqs->max_blocks_per_seq;
    p.max_partitions = 2;
    p.mode = pkv::kModeBalanced;
    p.min_chunk = pkv::kMinChunk;
    p.seg_cost = pkv::kSegCost;
    p.num_seqs = int32_t(list);
    p.q_len = item_width;
    p.context_lens = list_ctx;
    p.item_seq = list_seq;
    p.seq_start = list_start;
    p.row_map = list_rows;
    p.num_items = num_items;
    p.part_offset = 1;
    if ((st = attn_launch(p, cache, gqa, stream)) != PKV_OK) return st;
    pkv::ReduceParams r{};
    r.out = out;
    r.out_dtype = out_dtype;
    r.tmp_out = tmp_out;
    r.max_logits = max_logits;
    r.exp_sums = exp_sums;
    r.context_lens = seqs->context_lens;
    r.num_seqs = seqs->num_seqs;
    r.q_len = 1;
    r.num_heads = num_heads;
    r.head_dim = cache->head_dim;
    r.partition_size = 16;
    r.max_partitions = 2;
    r.seq_start = list_start + num_items;
    return cuda_result(pkv::launch_reduce(r, cs), "cascade reduce launch");
}

size_t pkv_sparse_workspace_bytes(int32_t num_seqs, int32_t num_kv_heads, int32_t head_dim, int32_t max_pages) {
    if (num_seqs < 0 || num_kv_heads < 1 || head_dim < 1 || max_pages < 0) return 0;
    return align256(size_t(num_seqs) * size_t(max_pages) * 4) + align256(size_t(num_seqs) * 4) +
           pkv::balanced_workspace_bytes(num_seqs, num_kv_heads, head_dim);
}

pkv_status pkv_paged_attention_sparse(void* out, pkv_dtype out_dtype, const void* q, pkv_dtype q_dtype,
                                      int32_t num_heads, float scale, const pkv_cache* cache, const pkv_seqs* seqs,
                                      const int32_t* page_lists, const int32_t* page_counts, int32_t max_pages,
                                      void* workspace, size_t workspace_bytes, uint32_t* err_flags,
                                      pkv_stream_t stream) {
    pkv::AttnParams p;
    int gqa = 0;
    pkv_status st = attn_setup(&p, q, q_dtype, num_heads, scale, cache, seqs, err_flags, &gqa);
    if (st != PKV_OK) return st;
    if (seqs->q_len != 1) return fail(PKV_ERR_UNSUPPORTED, "sparse page-indirection decode is for q_len 1");
    if (seqs->sliding_window != 0) return fail(PKV_ERR_UNSUPPORTED, "sparse page-indirection with a sliding window");
    if (max_pages < 1) return fail(PKV_ERR_INVALID_ARG, "max_pages %d", max_pages);
    if (!page_lists || !page_counts) return fail(PKV_ERR_INVALID_ARG, "page_lists / page_counts is NULL");
    if (int64_t(seqs->num_seqs) * max_pages > INT32_MAX / 2) return fail(PKV_ERR_INVALID_ARG, "page lists too large");
    if (seqs->num_seqs == 0) return ok();
    const size_t need = pkv_sparse_workspace_bytes(seqs->num_seqs, cache->num_kv_heads, cache->head_dim, max_pages);
    if (!workspace) return fail(PKV_ERR_INVALID_ARG, "workspace is NULL");
    if (workspace_bytes < need)
        return fail(PKV_ERR_INVALID_ARG, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
    uint8_t* w = static_cast<uint8_t*>(workspace);
    int32_t* table_c = reinterpret_cast<int32_t*>(w);
    w += align256(size_t(seqs->num_seqs) * size_t(max_pages) * 4);
    int32_t* ctx_c = reinterpret_cast<int32_t*>(w);
    w += align256(size_t(seqs->num_seqs) * 4);
    if ((st = balanced_setup(p, out, out_dtype, cache, seqs, w, need - size_t(w - static_cast<uint8_t*>(workspace)))) !=
        PKV_OK)
        return st;
    pkv::SparseParams sp{};
    sp.page_lists = page_lists;
    sp.page_counts = page_counts;
    sp.block_tables = seqs->block_tables;
    sp.context_lens = seqs->context_lens;
    sp.num_seqs = seqs->num_seqs;
    sp.max_pages = max_pages;
    sp.max_blocks = seqs->max_blocks_per_seq;
    sp.table_out = table_c;
    sp.ctx_out = ctx_c;
    sp.counters = p.counters;
    sp.num_counters = seqs->num_seqs * cache->num_kv_heads;
    sp.err = err_flags;
    cudaError_t e = pkv::launch_sparse_setup(sp, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_result(e, "sparse set-up launch");
    // the balanced attention over the compacted tables
    p.block_tables = table_c;
    p.context_lens = ctx_c;
    p.max_blocks = max_pages;
    p.partition_blocks = max_pages;
    p.wait_first = 1;
    return attn_launch(p, cache, gqa, stream);
}

int32_t pkv_sparse_worthwhile(const int32_t* page_counts, const int32_t* context_lens, int32_t num_seqs,
                              float min_sparsity) {
    if (!page_counts || !context_lens || num_seqs <= 0) return 0;
    long long listed = 0, total = 0;
    for (int s = 0; s < num_seqs; ++s) {
        const long long pages = context_lens[s] > 0 ? (context_lens[s] + 15) / 16 : 0;
        long long c = page_counts[s];
        c = c < 0 ? 0 : (c > pages ? pages : c);
        listed += c;
        total += pages;
    }
    if (total == 0) return 0;
    // min_sparsity arrives as a float: compare with a relative slack of 1e-6
    const double skipped = double(total - listed);
    return skipped >= double(min_sparsity) * double(total) * (1.0 - 1e-6) ? 1 : 0;
}

pkv_status pkv_decode_step_balanced(void* out, pkv_dtype out_dtype, const void* q, pkv_dtype q_dtype,
                                    int32_t num_heads, float scale, const pkv_cache* cache, const pkv_seqs* seqs,
                                    const void* k_new, const void* v_new, pkv_dtype src_dtype,
                                    const int64_t* slot_mapping, int32_t num_tokens, void* workspace,
                                    size_t workspace_bytes, uint32_t* err_flags, pkv_stream_t stream) {
    pkv::AttnParams p;
    int gqa = 0;
    pkv_status st = attn_setup(&p, q, q_dtype, num_heads, scale, cache, seqs, err_flags, &gqa);
    if (st != PKV_OK) return st;
    if (num_tokens < 0) return fail(PKV_ERR_INVALID_ARG, "num_tokens %d", num_tokens);
    if (cache->kind == PKV_CACHE_K8V4) {
        if (src_dtype != PKV_F16 && src_dtype != PKV_BF16) return fail(PKV_ERR_INVALID_ARG, "src_dtype %d", src_dtype);
    } else if (src_dtype != cache_dtype(cache)) {
        return fail(PKV_ERR_INVALID_ARG, "src_dtype must be the fp16/bf16 cache dtype");
    }
    if (num_tokens > 0) {
        CHECK_PTR(k_new, "k_new");
        CHECK_PTR(v_new, "v_new");
        if (!slot_mapping) return fail(PKV_ERR_INVALID_ARG, "slot_mapping is NULL");
    }
    if ((st = balanced_setup(p, out, out_dtype, cache, seqs, workspace, workspace_bytes)) != PKV_OK) return st;
    if (seqs->num_seqs == 0) {
        // nothing to attend: the write alone
        if (num_tokens == 0) return ok();
        return cache->kind == PKV_CACHE_K8V4
                   ? pkv_quantize_kv(cache, k_new, v_new, src_dtype, slot_mapping, num_tokens, err_flags, stream)
                   : pkv_reshape_and_cache(cache, k_new, v_new, slot_mapping, num_tokens, err_flags, stream);
    }
    p.kc = cache->k;
    p.vc = cache->v;
    p.k_new = k_new;
    p.v_new = v_new;
    p.slot_mapping = slot_mapping;
    p.num_new = num_tokens;
    p.src_dtype = src_dtype;
    return attn_launch(p, cache, gqa, stream);
}

}  // extern "C"

// ---------------------------------------------------------------- the allocation-free variant
// Scratch of pkv_paged_attention_balanced_noalloc: one array in the library's
// own device image, so a caller that cannot allocate device memory still gets
// the balanced schedule.  Every GPU that loads the library holds it until the
// process exits.  Host code must not use the symbol as a device address; the
// address is looked up with the caller's device current (noalloc_scratch).
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(PKV_NOALLOC_SCRATCH_BYTES);
static_assert(kNoAllocScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent from the driver, fetched once through the runtime.
CtxGetCurrentFn ctx_get_current_fn() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(f);
    });
    return fn;
}

// Device address of g_noalloc_scratch in the current context.  A call made
// while `stream` is not being captured looks the address up afresh
// (cudaGetSymbolAddress, with the caller's device current) and remembers it for
// that context; a call made during stream capture uses the remembered address,
// so the first call in a context must come before any capture.  Looking it up
// again on every uncaptured call keeps a cached address from outliving its
// module: after cudaDeviceReset, or in another context on the same device, the
// array sits at a different address.
void* noalloc_scratch(cudaStream_t stream, pkv_status* st) {
    constexpr int kSlots = 64;
    static std::mutex mu;
    static CUcontext ctxs[kSlots] = {};
    static void* addrs[kSlots] = {};
    static int next = 0;
    auto get_ctx = ctx_get_current_fn();
    if (!get_ctx) {
        *st = fail(PKV_ERR_CUDA, "cuCtxGetCurrent is unavailable from the driver");
        return nullptr;
    }
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        (void)cudaGetLastError();
        cap = cudaStreamCaptureStatusActive;   // treat an unanswerable query as capture: no look-up
    }
    std::lock_guard<std::mutex> lock(mu);
    if (cap == cudaStreamCaptureStatusNone) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            *st = fail(PKV_ERR_CUDA, "cudaGetSymbolAddress of the static scratch: %s", cudaGetErrorString(e));
            return nullptr;
        }
        CUcontext ctx = nullptr;
        if (get_ctx(&ctx) == CUDA_SUCCESS && ctx != nullptr) {
            int slot = -1;
            for (int i = 0; i < kSlots; ++i)
                if (ctxs[i] == ctx) slot = i;
            if (slot < 0) {
                slot = next;
                next = (next + 1) % kSlots;
                ctxs[slot] = ctx;
            }
            addrs[slot] = ptr;
        }
        return ptr;
    }
    CUcontext ctx = nullptr;
    if (get_ctx(&ctx) == CUDA_SUCCESS && ctx != nullptr)
        for (int i = 0; i < kSlots; ++i)
            if (ctxs[i] == ctx) return addrs[i];
    *st = fail(PKV_ERR_INVALID_ARG,
               "the first pkv_paged_attention_balanced_noalloc call in a context must come before stream capture "
               "(it looks up the static scratch's device address)");
    return nullptr;
}

}  // namespace

extern "C" {

pkv_status pkv_paged_attention_balanced_noalloc(void* out, pkv_dtype out_dtype, const void* q, pkv_dtype q_dtype,
                                                int32_t num_heads, float scale, const pkv_cache* cache,
                                                const pkv_seqs* seqs, uint32_t* err_flags, pkv_stream_t stream) {
    pkv::AttnParams p;
    int gqa = 0;
    pkv_status st = attn_setup(&p, q, q_dtype, num_heads, scale, cache, seqs, err_flags, &gqa);
    if (st != PKV_OK) return st;
    CHECK_PTR(out, "out");
    if (out_dtype != PKV_F16 && out_dtype != PKV_BF16 && out_dtype != PKV_F32)
        return fail(PKV_ERR_INVALID_ARG, "out_dtype %d", out_dtype);
    if (cache->num_kv_heads > pkv::kMaxGrid)
        return fail(PKV_ERR_UNSUPPORTED, "num_kv_heads %d above %d for the balanced schedule", cache->num_kv_heads,
                    pkv::kMaxGrid);
    if (seqs->num_seqs == 0) return ok();
    const size_t need = pkv::balanced_workspace_bytes(seqs->num_seqs, cache->num_kv_heads, cache->head_dim);
    if (need > kNoAllocScratchBytes)
        return fail(PKV_ERR_INVALID_ARG,
                    "batch too large for the static scratch: %d sequences x %d kv heads at head_dim %d need %zu "
                    "bytes, the library holds %zu (use pkv_paged_attention_balanced with your own workspace)",
                    seqs->num_seqs, cache->num_kv_heads, cache->head_dim, need, kNoAllocScratchBytes);
    void* ws = noalloc_scratch(reinterpret_cast<cudaStream_t>(stream), &st);
    if (!ws) return st;
    const size_t pairs = size_t(seqs->num_seqs) * size_t(cache->num_kv_heads);
    const size_t slots = size_t(pkv::kMaxGrid) + pairs;
    uint8_t* w = static_cast<uint8_t*>(ws);
    p.part_o = reinterpret_cast<float*>(w);
    w += align256(slots * 16 * size_t(cache->head_dim) * 4);
    p.part_ml = reinterpret_cast<float*>(w);
    w += align256(slots * 16 * 2 * 4);
    p.counters = reinterpret_cast<int32_t*>(w);
    // the array keeps whatever the previous call left: the piece counters must
    // start at zero (partials are always written before they are read)
    cudaError_t e = cudaMemsetAsync(p.counters, 0, pairs * sizeof(int32_t), reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_result(e, "clearing the static scratch counters");
    p.out = out;
    p.out_dtype = out_dtype;
    p.partition_blocks = seqs->max_blocks_per_seq;
    p.max_partitions = 1;
    p.mode = pkv::kModeBalanced;
    p.min_chunk = pkv::kMinChunk;
    p.seg_cost = pkv::kSegCost;
    return attn_launch(p, cache, gqa, stream);
}

pkv_status pkv_reduce(void* out, pkv_dtype out_dtype, const float* tmp_out, const float* max_logits,
                      const float* exp_sums, const pkv_seqs* seqs, int32_t num_heads, int32_t head_dim,
                      int32_t partition_size, int32_t max_partitions, pkv_stream_t stream) {
    pkv_status st = check_seqs(seqs);
    if (st != PKV_OK) return st;
    CHECK_PTR(out, "out");
    CHECK_PTR(tmp_out, "tmp_out");
    CHECK_PTR(max_logits, "max_logits");
    CHECK_PTR(exp_sums, "exp_sums");
    if (out_dtype != PKV_F16 && out_dtype != PKV_BF16 && out_dtype != PKV_F32)
        return fail(PKV_ERR_INVALID_ARG, "out_dtype %d", out_dtype);
    if (head_dim != 64 && head_dim != 128) return fail(PKV_ERR_UNSUPPORTED, "head_dim %d", head_dim);
    if (num_heads < 1) return fail(PKV_ERR_INVALID_ARG, "num_heads %d", num_heads);
    if (partition_size < 16 || partition_size % 16 != 0)
        return fail(PKV_ERR_INVALID_ARG, "partition_size %d", partition_size);
    if (max_partitions < 1) return fail(PKV_ERR_INVALID_ARG, "max_partitions %d", max_partitions);
    if (seqs->num_seqs == 0) return ok();
    if (int64_t(seqs->num_seqs) * seqs->q_len > INT32_MAX) return fail(PKV_ERR_INVALID_ARG, "too many rows");
    pkv::ReduceParams p{};
    p.out = out;
    p.out_dtype = out_dtype;
    p.tmp_out = tmp_out;
    p.max_logits = max_logits;
    p.exp_sums = exp_sums;
    p.context_lens = seqs->context_lens;
    p.num_seqs = seqs->num_seqs;
    p.q_len = seqs->q_len;
    p.num_heads = num_heads;
    p.head_dim = head_dim;
    p.partition_size = partition_size;
    p.max_partitions = max_partitions;
    p.window = seqs->sliding_window;
    return cuda_result(pkv::launch_reduce(p, reinterpret_cast<cudaStream_t>(stream)), "reduce launch");
}

pkv_status pkv_gather_kv_cache(void* k_out, void* v_out, const int32_t* cu_seq_lens, const pkv_cache* cache,
                               const pkv_seqs* seqs, uint32_t* err_flags, pkv_stream_t stream) {
    pkv_status st = check_cache(cache, true);
    if (st != PKV_OK) return st;
    if ((st = check_seqs(seqs)) != PKV_OK) return st;
    if (seqs->num_seqs == 0) return ok();
    CHECK_PTR(k_out, "k_out");
    CHECK_PTR(v_out, "v_out");
    if (!cu_seq_lens) return fail(PKV_ERR_INVALID_ARG, "cu_seq_lens is NULL");
    pkv::GatherParams p{};
    p.k_out = k_out;
    p.v_out = v_out;
    p.cu_seq_lens = cu_seq_lens;
    p.k_cache = cache->k;
    p.v_cache = cache->v;
    p.block_tables = seqs->block_tables;
    p.context_lens = seqs->context_lens;
    p.num_seqs = seqs->num_seqs;
    p.max_blocks = seqs->max_blocks_per_seq;
    p.num_blocks = cache->num_blocks;
    p.num_kv_heads = cache->num_kv_heads;
    p.head_dim = cache->head_dim;
    p.err = err_flags;
    return cuda_result(pkv::launch_gather(p, 2, reinterpret_cast<cudaStream_t>(stream)), "gather launch");
}

pkv_status pkv_gather_kv_cache_dequant(void* k_out, void* v_out, pkv_dtype out_dtype, const int32_t* cu_seq_lens,
                                       const pkv_cache* cache, const pkv_seqs* seqs, uint32_t* err_flags,
                                       pkv_stream_t stream) {
    pkv_status st = check_cache(cache, false);
    if (st != PKV_OK) return st;
    if (cache->kind != PKV_CACHE_K8V4) return fail(PKV_ERR_INVALID_ARG, "the dequantising gather needs a K8V4 cache");
    if (out_dtype != PKV_F16 && out_dtype != PKV_BF16) return fail(PKV_ERR_INVALID_ARG, "out_dtype %d", out_dtype);
    if ((st = check_seqs(seqs)) != PKV_OK) return st;
    if (seqs->num_seqs == 0) return ok();
    CHECK_PTR(k_out, "k_out");
    CHECK_PTR(v_out, "v_out");
    if (!cu_seq_lens) return fail(PKV_ERR_INVALID_ARG, "cu_seq_lens is NULL");
    pkv::GatherParams p{};
    p.k_out = k_out;
    p.v_out = v_out;
    p.cu_seq_lens = cu_seq_lens;
    p.k_cache = cache->k;
    p.v_cache = cache->v;
    p.k_scale = cache->k_scale;
    p.v_scale = cache->v_scale;
    p.v_zero = cache->v_zero;
    p.out_dtype = out_dtype;
    p.block_tables = seqs->block_tables;
    p.context_lens = seqs->context_lens;
    p.num_seqs = seqs->num_seqs;
    p.max_blocks = seqs->max_blocks_per_seq;
    p.num_blocks = cache->num_blocks;
    p.num_kv_heads = cache->num_kv_heads;
    p.head_dim = cache->head_dim;
    p.err = err_flags;
    return cuda_result(pkv::launch_gather_dequant(p, reinterpret_cast<cudaStream_t>(stream)),
                       "dequantising gather launch");
}

const char* pkv_status_string(pkv_status status) {
    switch (status) {
        case PKV_OK: return "ok";
        case PKV_ERR_INVALID_ARG: return "invalid argument";
        case PKV_ERR_UNSUPPORTED: return "unsupported shape or type";
        case PKV_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

const char* pkv_last_error(void) { return g_last_error.c_str(); }

}  // extern "C"
