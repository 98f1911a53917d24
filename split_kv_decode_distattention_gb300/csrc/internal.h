// Host-side declarations shared by the dattn translation units (not part of the public ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dattn.h"

namespace dattn {

constexpr int kConsumerWarps = 4;
constexpr int kAttnThreads = (kConsumerWarps + 1) * 32;
// Pipeline depth, a multiple of kConsumerWarps: consumer warp w takes the tiles k = w mod 4,
// so it has depth/4 - 1 tiles loading while it works on one. The 8-bit stages are half as
// large; 12 of them (48 KB for d = 128) keep more bytes in flight per warp without lowering
// the CTAs per SM, which 16 stages did for grouped heads. The 4-bit stages are a quarter as
// large; the 4-bit kernel runs four CTAs per SM (its consumers, not HBM, bound it, and more
// warps hide their latency), and 16 stages (32 KB) let the four fit in shared memory.
constexpr int kStagesBf16 = 8;
constexpr int kStagesF8 = 12;
constexpr int kStagesI4 = 16;
// The mixed pool's stages are 8-bit stages; a 4-bit tile fills half of one.
__host__ __device__ constexpr int attn_stages(int fmt) {
    return fmt == DATTN_KV_INT4 ? kStagesI4
         : (fmt == DATTN_KV_FP8_E4M3 || fmt == DATTN_KV_MIXED) ? kStagesF8
                                                                : kStagesBf16;
}
// Bytes of one K (or V) tile of 16 tokens in shared memory for a pool format (the mixed
// pool: the larger, 8-bit tile).
__host__ __device__ constexpr uint32_t attn_tile_bytes(int fmt, int D) {
    return (fmt == DATTN_KV_INT4 ? 8u
            : (fmt == DATTN_KV_FP8_E4M3 || fmt == DATTN_KV_MIXED) ? 16u
                                                                   : 32u) * (uint32_t)D;
}
constexpr int kMaxItems = 4096;     // B (or C) bound
constexpr int kMaxKvHeads = 256;
constexpr int kMaxGroup = 8;        // query heads per KV head
constexpr int kMaxTopK = 256;
constexpr int kMaxCtasPerSm = 4;    // bound used for workspace sizing with automatic splits
constexpr int32_t kSegCost = 6;     // cost units per segment in the balanced split

enum AttnMode : int { MODE_PARTIAL = 0, MODE_DENSE = 1, MODE_SPARSE = 2 };

// The per-KV-head formats of a mixed pool: bit h of i4 is set when KV head h is 4-bit (else
// 8-bit); h4 heads are 4-bit. A head's row within its region uses its index among the heads
// of its own format.
struct KvHeadFormats {
    int32_t h4;
    uint32_t i4[kMaxKvHeads / 32];
};
// Fills f from a layout (all-zero unless the layout is mixed); INVALID_ARG when a mixed
// layout's head_format is missing or names another format.
dattn_status_t head_formats(const dattn_kv_layout& L, KvHeadFormats& f);

__host__ __device__ __forceinline__ int32_t popc32(uint32_t x) {
#ifdef __CUDA_ARCH__
    return __popc(x);
#else
    return __builtin_popcount(x);
#endif
}
__host__ __device__ __forceinline__ bool head_is_i4(const KvHeadFormats& f, int32_t h) {
    return (f.i4[h >> 5] >> (h & 31)) & 1u;
}
// Index of KV head h among the heads of its own format.
__host__ __device__ __forceinline__ int32_t head_class_index(const KvHeadFormats& f, int32_t h,
                                                             bool i4) {
    int32_t n = 0;
    for (int32_t w = 0; w < (h >> 5); ++w) n += popc32(f.i4[w]);
    const uint32_t below = (h & 31) ? f.i4[h >> 5] & ((1u << (h & 31)) - 1u) : 0u;
    n += popc32(below);
    return i4 ? n : h - n;
}

// Everything one launch of the attention engine needs (device pointers unless noted).
struct AttnParams {
    int32_t mode;
    int32_t num_pages, Hkv, P, max_pages;
    const int32_t* block_table;
    const uint16_t* q;
    int32_t B, Hq, g;
    // query tokens per request (1 = decode; T > 1: multi-query decode, causal over the T
    // newest tokens) and the columns of a segment's tile, gq = g * T <= 8
    int32_t T, gq;
    float sl2;  // scale * log2(e)
    const int32_t* seq_lens;
    // dattn_partial
    int32_t C;
    const int32_t* chunk_req;
    const int32_t* chunk_indptr;
    const int32_t* chunk_pages;
    // block-sparse decode
    const int8_t* head_kind;
    int32_t sinks, local, top_k;
    const int32_t* selected;
    const int32_t* selected_phys;  // nullable: physical pages of `selected` (no table lookup)
    // fused one-token append (dattn_append_decode): the new token of request b is written at
    // position seq_lens[b] (quantized as the pool's format prescribes), attended by this
    // launch, and seq_lens[b] advances by one
    int32_t append;
    const uint16_t* k_new;  // [B][Hkv][D]
    const uint16_t* v_new;
    uint8_t* k_pool_w;      // the pools' bytes
    uint8_t* v_pool_w;
    float* kv_scale_w;      // the quantized pools' row scales
    uint16_t* stats;  // nullable: logical-page k_max / k_min
    int32_t* seq_lens_w;  // seq_lens, advanced by the launch
    // outputs: decode -> out [B][Hq][D], m_out / e_out [B][Hq] (nullable)
    //          partial -> out = MA [C][Hq][D], m_out / e_out [C][Hq]
    float* out;
    float* m_out;
    float* e_out;
    // workspace
    int32_t* counters;  // [nseg + 1]: per segment, then the append's arrival count
    float* slots;       // [(G + nseg)][slot_floats(g, D)]: MA [g][D], m [g], e [g], padding
    int32_t nseg;
    int32_t nitems;     // B for dense / sparse, C for partial
    int32_t* dev_err;
    // pool format (DATTN_KV_*). The 8-bit (FP8 E4M3) and 4-bit (symmetric integer) pools keep
    // one fp32 scale per (token, KV head) row; the scales of a 16-token tile are one 128-byte
    // run [16 K scales][16 V scales]
    int32_t fmt;
    const float* kv_scale;
    KvHeadFormats hf;  // DATTN_KV_MIXED: the per-head formats
};

// Floats of one workspace slot (a piece's partial): MA [g][D], then m [g] and e [g],
// padded to a multiple of four floats so that every slot starts on 16 bytes.
__host__ __device__ inline int32_t slot_floats(int32_t g, int32_t D) {
    return g * D + ((2 * g + 3) & ~3);
}

// Shared-memory layout of the attention engine, identical on host and device. A stage holds
// the K tile then the V tile of 16 tokens (bf16: 32*d bytes each; 8-bit: 16*d; 4-bit: 8*d);
// with a quantized pool, the stage's 16 K scales and 16 V scales sit in `scales`.
struct AttnSmem {
    uint32_t nstages, stage_bytes, stages, scales, bars, meta, flags, ws_m, ws_e, ws_o, kind_before,
        kinds, aplan, item_start, item_len, item_pos, qrow, scan, total;
};

// Integers of the head-aligned plan of a block-sparse launch (see the attention kernel):
// its scalars, then the retrieval and the streaming head lists.
constexpr int kAplanScalars = 8;

__host__ __device__ inline AttnSmem attn_smem_layout(int D, int g, int nitems, int Hkv,
                                                     bool sparse, int fmt, bool append = false) {
    AttnSmem s;
    const uint32_t ns = (uint32_t)attn_stages(fmt);
    s.nstages = ns;
    s.stage_bytes = 2u * attn_tile_bytes(fmt, D);
    uint32_t o = 0;
    s.stages = o;      o += ns * s.stage_bytes;
    s.scales = o;      o += fmt != DATTN_KV_BF16 ? ns * 128u : 0u;
    s.bars = o;        o += 2u * ns * 8u;
    s.meta = o;        o += ns * 4u;
    s.flags = o;       o += 32u;  // abort flag, last flag, then 5 plan constants
    s.ws_m = o;        o += kConsumerWarps * kMaxGroup * 4u;
    s.ws_e = o;        o += kConsumerWarps * kMaxGroup * 4u;
    s.ws_o = o;        o += (uint32_t)(kConsumerWarps * g * D) * 4u;
    s.kind_before = o; o += sparse ? (uint32_t)(Hkv + 1) * 3u * 4u : 0u;
    s.kinds = o;       o += sparse ? (uint32_t)Hkv * 4u : 0u;
    s.aplan = o;       o += sparse ? (uint32_t)(kAplanScalars + 2 * Hkv) * 4u : 0u;
    o = (o + 15u) & ~15u;
    s.item_start = o;  o += (uint32_t)(nitems + 1) * 4u;
    s.item_len = o;    o += (uint32_t)nitems * 4u;
    s.item_pos = o;    o += append ? (uint32_t)nitems * 4u : 0u;
    o = (o + 15u) & ~15u;
    // fused append to a quantized pool: each consumer lane's codes and scale of the new row
    s.qrow = o;        o += (append && fmt != DATTN_KV_BF16) ? kConsumerWarps * 32u * 3u * 4u : 0u;
    s.scan = o;        o += 8u * 4u;
    s.total = o + 1024u;  // slack to align the dynamic base to 1024 bytes
    return s;
}

// Device properties and cached driver entry points.
int sm_count_current();
dattn_status_t make_kv_tensor_map(void* tmap_out, const void* pool, int64_t rows, int D);
// 2-D map over rows of `row_bytes` one-byte elements (8-bit codes: d; packed 4-bit codes:
// d / 2), one box of 16 rows, swizzled by the row size (128, 64 or 32 bytes).
dattn_status_t make_kv_tensor_map_u8(void* tmap_out, const void* pool, int64_t rows,
                                     int row_bytes);

dattn_status_t launch_attention(const AttnParams& p, const void* k_pool, const void* v_pool,
                                int D, int32_t num_splits, void* ws, size_t ws_bytes,
                                cudaStream_t stream, int64_t tiles_bound);

// Launches kernel<<<grid, block, smem, stream>>>(args...) with programmatic stream
// serialization, so that its launch and prologue overlap the previous kernel on the stream.
// Every kernel launched this way calls grid_dependency_wait() before reading data that an
// earlier kernel may write.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Number of CTAs for a launch with an upper bound of total_tiles tiles.
int32_t choose_splits(int64_t total_tiles, int32_t requested, int occupancy);

// Bytes of the workspace's counter region: one counter per segment and the append's arrival
// counter, padded to 256 bytes. The partial slots follow it.
inline size_t attn_counter_bytes(int32_t nseg) {
    return ((size_t)(nseg + 1) * 4 + 255) & ~(size_t)255;
}
size_t attn_workspace_bytes(int32_t nseg, int32_t g, int32_t D, int32_t G);
size_t select_workspace_bytes(int32_t nseg, int32_t top_k, int32_t G);

}  // namespace dattn
