// The extern "C" entry points of libdattn.so: host-side validation, then dispatch to the
// kernels. Nothing here allocates, frees or synchronises. See include/dattn.h for the
// contract of every call.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dattn {

dattn_status_t launch_merge(int32_t B, int32_t C, int32_t Hq, int32_t D, const int32_t* indptr,
                            int32_t R, const float* m, const float* e, const float* MA,
                            float* out, float* m_g, float* e_g, float* MA_g, int32_t* dev_err,
                            cudaStream_t stream);
dattn_status_t launch_kv_append(const dattn_kv_layout& L, void* k_pool, void* v_pool,
                                uint16_t* stats, const uint16_t* k_new, const uint16_t* v_new,
                                int32_t B, int32_t T, int32_t* seq_lens, int32_t* dev_err,
                                cudaStream_t stream);
dattn_status_t launch_page_select(const dattn_kv_layout& Lay, const uint16_t* stats,
                                  const uint16_t* q, int32_t B, int32_t Hq,
                                  const int32_t* seq_lens, const int8_t* head_kind,
                                  int32_t top_k, int32_t* selected, int32_t* selected_phys,
                                  void* ws, size_t ws_bytes, int32_t num_splits,
                                  int32_t* dev_err, cudaStream_t stream, int64_t units_bound);

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks shared by every call that reads the pool.
dattn_status_t check_layout(const dattn_kv_layout* L) {
    if (L == nullptr || L->block_table == nullptr) return DATTN_ERR_INVALID_ARG;
    if (L->num_pages <= 0 || L->num_kv_heads <= 0 || L->max_pages_per_req <= 0 ||
        L->page_size <= 0 || L->head_dim <= 0)
        return DATTN_ERR_INVALID_ARG;
    if (L->head_dim != 64 && L->head_dim != 128) return DATTN_ERR_UNSUPPORTED;
    if (L->page_size % 16 != 0 || L->page_size > 256) return DATTN_ERR_UNSUPPORTED;
    if (L->num_kv_heads > kMaxKvHeads) return DATTN_ERR_UNSUPPORTED;
    // TMA row coordinates and token positions are 32-bit
    if ((int64_t)L->num_pages * L->num_kv_heads * L->page_size >= (1ll << 31))
        return DATTN_ERR_UNSUPPORTED;
    if ((int64_t)L->max_pages_per_req * L->page_size >= (1ll << 30)) return DATTN_ERR_UNSUPPORTED;
    if (L->kv_format != DATTN_KV_BF16 && L->kv_format != DATTN_KV_FP8_E4M3 &&
        L->kv_format != DATTN_KV_INT4 && L->kv_format != DATTN_KV_MIXED)
        return DATTN_ERR_INVALID_ARG;
    if (L->kv_format != DATTN_KV_BF16 && (!L->kv_scale || !aligned16(L->kv_scale)))
        return DATTN_ERR_INVALID_ARG;
    KvHeadFormats f;
    return head_formats(*L, f);
}

dattn_status_t check_heads(const dattn_kv_layout* L, int32_t B, int32_t Hq) {
    if (B < 0 || Hq <= 0) return DATTN_ERR_INVALID_ARG;
    if (Hq % L->num_kv_heads != 0) return DATTN_ERR_INVALID_ARG;
    if (Hq / L->num_kv_heads > kMaxGroup) return DATTN_ERR_UNSUPPORTED;
    if (B > kMaxItems) return DATTN_ERR_UNSUPPORTED;
    return DATTN_OK;
}

}  // namespace

dattn_status_t head_formats(const dattn_kv_layout& L, KvHeadFormats& f) {
    f = KvHeadFormats{};
    if (L.kv_format != DATTN_KV_MIXED) return DATTN_OK;
    if (L.head_format == nullptr) return DATTN_ERR_INVALID_ARG;
    for (int32_t h = 0; h < L.num_kv_heads; ++h) {
        const int8_t v = L.head_format[h];
        if (v != DATTN_KV_FP8_E4M3 && v != DATTN_KV_INT4) return DATTN_ERR_INVALID_ARG;
        if (v == DATTN_KV_INT4) {
            f.i4[h >> 5] |= 1u << (h & 31);
            ++f.h4;
        }
    }
    return DATTN_OK;
}

int sm_count_current() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
    int n = g_sm_count[dev].load(std::memory_order_relaxed);
    if (n <= 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            return 1;
        g_sm_count[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

int32_t choose_splits(int64_t total_tiles, int32_t requested, int occupancy) {
    if (requested > 0) return requested > (1 << 20) ? (1 << 20) : requested;
    int occ = occupancy < 1 ? 1 : (occupancy > kMaxCtasPerSm ? kMaxCtasPerSm : occupancy);
    int64_t G = (int64_t)sm_count_current() * occ;
    const int64_t cap = total_tiles / 16 > 1 ? total_tiles / 16 : 1;
    if (G > cap) G = cap;
    return G < 1 ? 1 : (int32_t)G;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D map over a pool of codes seen as rows of row_bytes bytes (8-bit: d; packed 4-bit:
// d / 2): one box {row_bytes, 16} is a 16-token row group of one (page, KV head), landing as
// [row][row_bytes] with the swizzle of the row's size (128, 64 or 32 bytes), which keeps
// ldmatrix conflict-free.
dattn_status_t make_kv_tensor_map_u8(void* tmap_out, const void* pool, int64_t rows,
                                     int row_bytes) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return DATTN_ERR_CUDA;
    if (row_bytes != 128 && row_bytes != 64 && row_bytes != 32) return DATTN_ERR_UNSUPPORTED;
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)row_bytes, 16};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle swz = row_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                   : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                     : CU_TENSOR_MAP_SWIZZLE_32B;
    CUresult r = fn(static_cast<CUtensorMap*>(tmap_out), CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                    const_cast<void*>(pool), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DATTN_OK : DATTN_ERR_CUDA;
}

// 3-D map over the pool seen as rows of d bf16 values, split into 128-byte halves:
// dim0 = 64 values of one half (contiguous), dim1 = row (stride d*2 bytes), dim2 = half
// (stride 128 bytes). One box {64, 16, d/64} is a whole 16-token row group of one (page, KV
// head). It lands in shared memory as [half][row][64 values] with the 128-byte swizzle,
// which keeps ldmatrix conflict-free. One TMA instruction moves the whole K (or V) tile.
dattn_status_t make_kv_tensor_map(void* tmap_out, const void* pool, int64_t rows, int D) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (fn == nullptr) return DATTN_ERR_CUDA;
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(D / 64)};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, 128};
    cuuint32_t box[3] = {64, 16, (cuuint32_t)(D / 64)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(static_cast<CUtensorMap*>(tmap_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                    const_cast<void*>(pool), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DATTN_OK : DATTN_ERR_CUDA;
}

}  // namespace dattn

using namespace dattn;

extern "C" {

const char* dattn_version(void) { return "dattn 0.1.0 sm_103a"; }

const char* dattn_status_string(dattn_status_t s) {
    switch (s) {
        case DATTN_OK: return "DATTN_OK";
        case DATTN_ERR_INVALID_ARG: return "DATTN_ERR_INVALID_ARG";
        case DATTN_ERR_UNSUPPORTED: return "DATTN_ERR_UNSUPPORTED";
        case DATTN_ERR_WORKSPACE: return "DATTN_ERR_WORKSPACE";
        case DATTN_ERR_CUDA: return "DATTN_ERR_CUDA";
    }
    return "DATTN_UNKNOWN_STATUS";
}

void dattn_split_range(int64_t total_tiles, int32_t num_splits, int32_t cta, int64_t* begin,
                       int64_t* end) {
    if (begin == nullptr || end == nullptr) return;
    if (num_splits <= 0 || cta < 0 || cta >= num_splits || total_tiles < 0) {
        *begin = *end = 0;
        return;
    }
    *begin = split_begin(total_tiles, num_splits, cta);
    *end = split_begin(total_tiles, num_splits, cta + 1);
}

int32_t dattn_split_owner(int64_t tile, int64_t total_tiles, int32_t num_splits) {
    if (num_splits <= 0 || total_tiles <= 0 || tile < 0 || tile >= total_tiles) return -1;
    return split_owner(tile, total_tiles, num_splits);
}

int32_t dattn_auto_splits(int64_t total_tiles) {
    return choose_splits(total_tiles, 0, kMaxCtasPerSm);
}

size_t dattn_workspace_size(int32_t items, int32_t Hq, int32_t Hkv, int32_t head_dim,
                            int32_t top_k, int32_t num_splits) {
    if (items < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || top_k < 0 || num_splits < 0)
        return 0;
    if (head_dim != 64 && head_dim != 128) return 0;
    const int32_t nseg = items * Hkv;
    const int32_t G = num_splits > 0 ? num_splits : sm_count_current() * kMaxCtasPerSm;
    size_t bytes = attn_workspace_bytes(nseg, Hq / Hkv, head_dim, G);
    if (top_k > 0) {
        const size_t sel = select_workspace_bytes(nseg, top_k, G);
        if (sel > bytes) bytes = sel;
    }
    return bytes;
}

dattn_status_t dattn_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    if (ws == nullptr && ws_bytes > 0) return DATTN_ERR_INVALID_ARG;
    if (ws_bytes == 0) return DATTN_OK;
    return cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? DATTN_OK
               : DATTN_ERR_CUDA;
}

dattn_status_t dattn_kv_append(const dattn_kv_layout* layout, void* k_pool,
                               void* v_pool, dattn_bf16* stats, const dattn_bf16* k_new,
                               const dattn_bf16* v_new, int32_t B, int32_t T,
                               int32_t* seq_lens, int32_t* dev_err, void* stream) {
    dattn_status_t st = check_layout(layout);
    if (st != DATTN_OK) return st;
    if (B < 0 || T < 0) return DATTN_ERR_INVALID_ARG;
    if (B == 0 || T == 0) return DATTN_OK;
    if (!k_pool || !v_pool || !k_new || !v_new || !seq_lens) return DATTN_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(k_new) || !aligned16(v_new) ||
        (stats && !aligned16(stats)))
        return DATTN_ERR_INVALID_ARG;
    if ((int64_t)B * T >= (1ll << 31) / 8) return DATTN_ERR_UNSUPPORTED;
    if (B > 65535) return DATTN_ERR_UNSUPPORTED;
    return launch_kv_append(*layout, k_pool, v_pool, stats, k_new, v_new, B, T, seq_lens, dev_err,
                            static_cast<cudaStream_t>(stream));
}

dattn_status_t dattn_partial(const dattn_kv_layout* layout, const void* k_pool,
                             const void* v_pool, const dattn_bf16* q, int32_t B,
                             int32_t Hq, float scale, const int32_t* seq_lens, int32_t C,
                             const int32_t* chunk_req, const int32_t* chunk_page_indptr,
                             const int32_t* chunk_pages, float* m, float* e, float* MA,
                             void* ws, size_t ws_bytes, int32_t num_splits, int32_t* dev_err,
                             void* stream) {
    dattn_status_t st = check_layout(layout);
    if (st != DATTN_OK) return st;
    if ((st = check_heads(layout, B, Hq)) != DATTN_OK) return st;
    if (C < 0 || num_splits < 0) return DATTN_ERR_INVALID_ARG;
    if (C > kMaxItems) return DATTN_ERR_UNSUPPORTED;
    if (C == 0) return DATTN_OK;
    if (!k_pool || !v_pool || !q || !seq_lens || !chunk_req || !chunk_page_indptr ||
        !chunk_pages || !m || !e || !MA)
        return DATTN_ERR_INVALID_ARG;
    if (B == 0) return DATTN_ERR_INVALID_ARG;  // chunks must name a request
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(q)) return DATTN_ERR_INVALID_ARG;
    const int64_t bound = (int64_t)C * layout->num_kv_heads *
                          ((int64_t)layout->max_pages_per_req * (layout->page_size / 16) + kSegCost);
    if (bound >= (1ll << 31)) return DATTN_ERR_UNSUPPORTED;
    AttnParams p{};
    p.mode = MODE_PARTIAL;
    p.num_pages = layout->num_pages;
    p.Hkv = layout->num_kv_heads;
    p.P = layout->page_size;
    p.max_pages = layout->max_pages_per_req;
    p.block_table = layout->block_table;
    p.q = q;
    p.B = B;
    p.Hq = Hq;
    p.g = Hq / p.Hkv;
    p.T = 1;
    p.gq = p.g;
    p.sl2 = scale * kLog2e;
    p.seq_lens = seq_lens;
    p.C = C;
    p.chunk_req = chunk_req;
    p.chunk_indptr = chunk_page_indptr;
    p.chunk_pages = chunk_pages;
    p.out = MA;
    p.m_out = m;
    p.e_out = e;
    p.nseg = C * p.Hkv;
    p.nitems = C;
    p.dev_err = dev_err;
    p.fmt = layout->kv_format;
    p.kv_scale = layout->kv_scale;
    head_formats(*layout, p.hf);  // checked with the layout
    return launch_attention(p, k_pool, v_pool, layout->head_dim, num_splits, ws, ws_bytes,
                            static_cast<cudaStream_t>(stream), bound);
}

dattn_status_t dattn_merge(int32_t B, int32_t C, int32_t Hq, int32_t head_dim,
                           const int32_t* chunk_indptr, const float* m, const float* e,
                           const float* MA, float* out, float* m_g, float* e_g, float* MA_g,
                           int32_t* dev_err, void* stream) {
    if (B < 0 || C < 0 || Hq <= 0) return DATTN_ERR_INVALID_ARG;
    if (head_dim <= 0 || head_dim > 128) return DATTN_ERR_UNSUPPORTED;
    if (B == 0) return DATTN_OK;
    if (B > 65535) return DATTN_ERR_UNSUPPORTED;
    if (!chunk_indptr) return DATTN_ERR_INVALID_ARG;
    if (C > 0 && (!m || !e || !MA)) return DATTN_ERR_INVALID_ARG;
    return launch_merge(B, C, Hq, head_dim, chunk_indptr, 0, m, e, MA, out, m_g, e_g, MA_g,
                        dev_err, static_cast<cudaStream_t>(stream));
}

dattn_status_t dattn_merge_gathered(int32_t B, int32_t R, int32_t Hq, int32_t head_dim,
                                    const float* m, const float* e, const float* MA, float* out,
                                    float* m_g, float* e_g, float* MA_g, int32_t* dev_err,
                                    void* stream) {
    if (B < 0 || R < 0 || Hq < 0) return DATTN_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128) return DATTN_ERR_UNSUPPORTED;
    if (B > kMaxItems || (int64_t)R * B > (1ll << 30)) return DATTN_ERR_UNSUPPORTED;
    if (B == 0 || Hq == 0) return DATTN_OK;
    if (R > 0 && (!m || !e || !MA)) return DATTN_ERR_INVALID_ARG;
    return launch_merge(B, R * B, Hq, head_dim, nullptr, R, m, e, MA, out, m_g, e_g, MA_g,
                        dev_err, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// The fused append of dattn_append_decode (k_new != NULL): the pool, statistics and lengths
// it writes.
struct AppendArgs {
    void* k_pool;
    void* v_pool;
    dattn_bf16* stats;
    const dattn_bf16* k_new;
    const dattn_bf16* v_new;
    int32_t* seq_lens;
};

// The fused decode of dattn_decode (T = 1), dattn_decode_multi (T query tokens) and
// dattn_append_decode (T = 1 with app != NULL).
dattn_status_t decode_impl(const dattn_kv_layout* layout, const void* k_pool, const void* v_pool,
                           const dattn_bf16* q, int32_t B, int32_t T, int32_t Hq, float scale,
                           const int32_t* seq_lens, const dattn_sparse* sparse,
                           int32_t num_splits, void* ws, size_t ws_bytes, float* out, float* m_g,
                           float* e_g, int32_t* dev_err, void* stream,
                           const AppendArgs* app = nullptr) {
    dattn_status_t st = check_layout(layout);
    if (st != DATTN_OK) return st;
    if ((st = check_heads(layout, B, Hq)) != DATTN_OK) return st;
    if (num_splits < 0 || T < 1) return DATTN_ERR_INVALID_ARG;
    if ((Hq / layout->num_kv_heads) * (int64_t)T > kMaxGroup) return DATTN_ERR_UNSUPPORTED;
    if (T > 1 && sparse != nullptr) return DATTN_ERR_UNSUPPORTED;
    if (B == 0) return DATTN_OK;
    if (!k_pool || !v_pool || !q || !seq_lens || !out) return DATTN_ERR_INVALID_ARG;
    if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(q)) return DATTN_ERR_INVALID_ARG;
    if (app != nullptr) {
        if (!app->k_new || !app->v_new) return DATTN_ERR_INVALID_ARG;
        if (!aligned16(app->k_new) || !aligned16(app->v_new) ||
            (app->stats && !aligned16(app->stats)))
            return DATTN_ERR_INVALID_ARG;
    }
    const int32_t per_page = layout->page_size / 16;
    const int64_t dense_tiles = (int64_t)layout->max_pages_per_req * per_page;
    int64_t per_head = dense_tiles;
    AttnParams p{};
    p.mode = MODE_DENSE;
    if (sparse != nullptr) {
        if (!sparse->head_kind || sparse->sinks < 0 || sparse->local < 0 || sparse->top_k < 0)
            return DATTN_ERR_INVALID_ARG;
        if (sparse->top_k > kMaxTopK || sparse->sinks > (1 << 20) || sparse->local > (1 << 20))
            return DATTN_ERR_UNSUPPORTED;
        if (sparse->top_k > 0 && !sparse->selected) return DATTN_ERR_INVALID_ARG;
        p.mode = MODE_SPARSE;
        p.head_kind = sparse->head_kind;
        p.sinks = sparse->sinks;
        p.local = sparse->local;
        p.top_k = sparse->top_k;
        p.selected = sparse->selected;
        p.selected_phys = sparse->selected_phys;
        const int64_t retr = (int64_t)sparse->top_k * per_page;
        const int64_t strm = (sparse->sinks + 15) / 16 + (sparse->local + 15) / 16 + 1;
        if (retr > per_head) per_head = retr;
        if (strm > per_head) per_head = strm;
    }
    const int64_t bound = (int64_t)B * layout->num_kv_heads * (per_head + kSegCost);
    if (bound >= (1ll << 31)) return DATTN_ERR_UNSUPPORTED;
    p.num_pages = layout->num_pages;
    p.Hkv = layout->num_kv_heads;
    p.P = layout->page_size;
    p.max_pages = layout->max_pages_per_req;
    p.block_table = layout->block_table;
    p.q = q;
    p.B = B;
    p.Hq = Hq;
    p.g = Hq / p.Hkv;
    p.T = T;
    p.gq = p.g * T;
    p.sl2 = scale * kLog2e;
    p.seq_lens = seq_lens;
    p.out = out;
    p.m_out = m_g;
    p.e_out = e_g;
    p.nseg = B * p.Hkv;
    p.nitems = B;
    p.dev_err = dev_err;
    p.fmt = layout->kv_format;
    p.kv_scale = layout->kv_scale;
    head_formats(*layout, p.hf);  // checked with the layout
    if (app != nullptr) {
        p.append = 1;
        p.k_new = app->k_new;
        p.v_new = app->v_new;
        p.k_pool_w = static_cast<uint8_t*>(app->k_pool);
        p.v_pool_w = static_cast<uint8_t*>(app->v_pool);
        p.kv_scale_w = layout->kv_scale;
        p.stats = app->stats;
        p.seq_lens_w = app->seq_lens;
    }
    return launch_attention(p, k_pool, v_pool, layout->head_dim, num_splits, ws, ws_bytes,
                            static_cast<cudaStream_t>(stream), bound);
}

}  // namespace

extern "C" {

dattn_status_t dattn_decode(const dattn_kv_layout* layout, const void* k_pool,
                            const void* v_pool, const dattn_bf16* q, int32_t B,
                            int32_t Hq, float scale, const int32_t* seq_lens,
                            const dattn_sparse* sparse, int32_t num_splits, void* ws,
                            size_t ws_bytes, float* out, float* m_g, float* e_g,
                            int32_t* dev_err, void* stream) {
    return decode_impl(layout, k_pool, v_pool, q, B, 1, Hq, scale, seq_lens, sparse, num_splits,
                       ws, ws_bytes, out, m_g, e_g, dev_err, stream);
}

dattn_status_t dattn_append_decode(const dattn_kv_layout* layout, void* k_pool, void* v_pool,
                                   dattn_bf16* stats, const dattn_bf16* k_new,
                                   const dattn_bf16* v_new, const dattn_bf16* q, int32_t B,
                                   int32_t Hq, float scale, int32_t* seq_lens,
                                   const dattn_sparse* sparse, int32_t num_splits, void* ws,
                                   size_t ws_bytes, float* out, float* m_g, float* e_g,
                                   int32_t* dev_err, void* stream) {
    const AppendArgs app{k_pool, v_pool, stats, k_new, v_new, seq_lens};
    return decode_impl(layout, k_pool, v_pool, q, B, 1, Hq, scale, seq_lens, sparse, num_splits,
                       ws, ws_bytes, out, m_g, e_g, dev_err, stream, &app);
}

dattn_status_t dattn_decode_multi(const dattn_kv_layout* layout, const void* k_pool,
                                  const void* v_pool, const dattn_bf16* q, int32_t B, int32_t T,
                                  int32_t Hq, float scale, const int32_t* seq_lens,
                                  int32_t num_splits, void* ws, size_t ws_bytes, float* out,
                                  float* m_g, float* e_g, int32_t* dev_err, void* stream) {
    return decode_impl(layout, k_pool, v_pool, q, B, T, Hq, scale, seq_lens, nullptr, num_splits,
                       ws, ws_bytes, out, m_g, e_g, dev_err, stream);
}

dattn_status_t dattn_page_select(const dattn_kv_layout* layout, const dattn_bf16* stats,
                                 const dattn_bf16* q, int32_t B, int32_t Hq,
                                 const int32_t* seq_lens, const int8_t* head_kind,
                                 int32_t top_k, int32_t* selected, int32_t* selected_phys,
                                 void* ws, size_t ws_bytes, int32_t num_splits,
                                 int32_t* dev_err, void* stream) {
    dattn_status_t st = check_layout(layout);
    if (st != DATTN_OK) return st;
    if ((st = check_heads(layout, B, Hq)) != DATTN_OK) return st;
    if (top_k < 0 || num_splits < 0) return DATTN_ERR_INVALID_ARG;
    if (top_k > kMaxTopK) return DATTN_ERR_UNSUPPORTED;
    const int32_t lpg = layout->page_size / 16;  // logical pages per physical page
    if (lpg & (lpg - 1)) return DATTN_ERR_UNSUPPORTED;
    if (B == 0 || top_k == 0) return DATTN_OK;
    if (!stats || !q || !seq_lens || !head_kind || !selected) return DATTN_ERR_INVALID_ARG;
    if (!aligned16(stats)) return DATTN_ERR_INVALID_ARG;
    const int64_t bound = (int64_t)B * layout->num_kv_heads * layout->max_pages_per_req;
    if (bound * 4 >= (1ll << 31)) return DATTN_ERR_UNSUPPORTED;
    return launch_page_select(*layout, stats, q, B, Hq, seq_lens, head_kind, top_k, selected,
                              selected_phys, ws, ws_bytes, num_splits, dev_err,
                              static_cast<cudaStream_t>(stream), bound);
}

}  // extern "C"
