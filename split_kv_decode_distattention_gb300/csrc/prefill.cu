// Block-sparse prefill (dattn_prefill): a chunk of Tq new query tokens per request attends
// the paged cache causally, key block by key block.
//
// "LLM长序列服务优化：LServe的块稀疏注意力技术": §2.1.1 cuts the KV history into fixed
// 64-token blocks and loads and computes only the chosen ones; §2.1.2 gives streaming heads a
// static Lambda pattern (the initial blocks plus the blocks next to the query) and retrieval
// heads a set of blocks chosen at run time; §2.2.1 walks the chosen blocks with a block
// iterator, so the compute loop has no branches on the mask.
//
// GB300 design: the contraction runs on the 5th-generation tensor cores. One CTA takes 128
// query rows: one 64-token query block of two query heads of a KV head when the group is
// even (both halves keep the same key blocks), else two query blocks of one query head. The
// heads of a KV head are neighbouring CTAs, so their K/V reads meet in L2. KV heads run in
// groups, each group's last rows (the most key blocks under the causal mask) first: a group
// is one KV head when its tiles fill three waves, so the K/V in flight stays in L2, else as
// many KV heads as it takes to fill them, so no long tile starts late. The key blocks each
// half keeps are built into shared-memory bitmaps, and every role walks their union in the
// same order: the block iterator. Seven warps:
//   - two producer warps, one for K and one for V, stream each key block's four 16-token
//     tiles by TMA (as [d/64 halves][64 rows][128 B] with the 128-byte swizzle, one box per
//     half and tile) into a two-stage K ring and a three-stage V ring; each resolves the
//     pages of eight blocks at once, one lane per tile, and the K warp also publishes each
//     block's metadata (index, which half keeps it, tile lengths);
//   - one thread issues tcgen05.mma: S = Q K^T (M 128, N 64, K d; Q and K from shared
//     memory, fp32 accumulator in tensor memory, double-buffered so the next block's scores
//     are computed during this block's softmax), then O += P V (M 128, N d, K 64; P from
//     tensor memory, V from shared memory as an MN-major operand), and commits each to an
//     mbarrier; K's stage is released when S is done, V's when P V is;
//   - four warps hold one query row per thread: they read the row's 64 scores from tensor
//     memory, mask them (the row's half keeps the block, the key is written and at or before
//     the query), keep the online softmax in base 2 on packed fp32 pairs and write P back
//     into the score buffer as two bf16 terms (hi: p cut to 16 bits; lo: the rest, rounded),
//     which the PV product reads.
// O is rescaled lazily, only when a row's maximum grows by more than 2^8, so most blocks touch
// tensor memory only through the products. No CTA depends on another: no workspace, no merge.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dattn {

namespace {

#define kPfNegInf (-__int_as_float(0x7f800000))

constexpr int kPfBlock = 64;                       // query and key block, tokens
constexpr int kPfTiles = kPfBlock / 16;            // tiles per key block

struct PfParams {
    int32_t num_pages, Hkv, P, max_pages;
    const int32_t* block_table;
    const uint16_t* q;
    int32_t B, Tq, Hq, g;
    float sl2;  // scale * log2(e)
    const int32_t* seq_lens;
    int32_t nqb;  // 128-row tiles per (request, head slot) a chunk can touch
    // 1: a CTA's 128 rows are one 64-token query block of two query heads of one KV head
    // (even g; both halves keep the same key blocks); 0: two query blocks of one query head
    int32_t head_pairs;
    int32_t kv_group;  // KV heads whose tiles run together (a divisor of Hkv)
    // block sparsity (head_kind == nullptr: dense causal)
    const int8_t* head_kind;
    int32_t sink_blocks, local_blocks, max_sel, qblock_stride;
    const int32_t* block_lists;
    float* out;
    float* m_out;
    float* e_out;
    int32_t* dev_err;
};

__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// ------------------------------------------------------------------ tcgen05 prefill

constexpr int kTcRows = 128;         // query rows per CTA (M of both products)
constexpr int kTcSoftWarps = 4;      // one thread per row
constexpr int kTcProdWarp = 4;       // TMA producer of K (and the block metadata)
constexpr int kTcMmaWarp = 5;        // tcgen05.mma issuer
constexpr int kTcVWarp = 6;          // TMA producer of V
constexpr int kTcThreads = 7 * 32;
constexpr int kTcKStages = 2;        // K blocks in flight (also the two score buffers)
constexpr int kTcVStages = 3;        // V blocks in flight
constexpr int kTcMetaSlots = 4;      // per-block metadata slots (block j in slot j % 4)
constexpr int kTcBars = 20;          // mbarriers of the pipeline
constexpr uint32_t kTcCols = 256;    // TMEM: O [0, 128), S0 [128, 192), S1 [192, 256)
constexpr float kTcRescale = 8.f;    // lazy rescale threshold (log2 units)

__device__ __forceinline__ void tc_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D (TMEM) (+)= A (smem descriptor) * B (smem descriptor)
__device__ __forceinline__ void tc_mma_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D (TMEM) (+)= A (TMEM) * B (smem descriptor)
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives once on the mbarrier when every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// 32 consecutive TMEM columns of this thread's lane (the warp's 32 lanes at once)
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
        "%28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// Packed fp32 pairs (Blackwell's two-wide fp32 FMA and add)
__device__ __forceinline__ uint64_t pack_f32x2(float a, float b) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
// (r0, r1) = (x0, x1) * m + c, m and c packed pairs, each lane rounded once
__device__ __forceinline__ void fma_f32x2(float x0, float x1, uint64_t m, uint64_t c, float& r0,
                                          float& r1) {
    asm("{\n\t.reg .b64 a, d;\n\tmov.b64 a, {%2, %3};\n\tfma.rn.f32x2 d, a, %4, %5;\n\t"
        "mov.b64 {%0, %1}, d;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "f"(x0), "f"(x1), "l"(m), "l"(c));
}
// (a0, a1) += (b0, b1)
__device__ __forceinline__ void add_f32x2(float& a0, float& a1, float b0, float b1) {
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%0, %1};\n\tmov.b64 b, {%2, %3};\n\t"
        "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "+f"(a0), "+f"(a1)
        : "f"(b0), "f"(b1));
}
// (r0, r1) = (a0, a1) - (b0, b1)
__device__ __forceinline__ void sub_f32x2(float a0, float a1, float b0, float b1, float& r0,
                                          float& r1) {
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "sub.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(r0), "=f"(r1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
// max(a, b, c) in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
// maximum of 64 values over eight independent chains of three-input maxima
__device__ __forceinline__ float row_max64(const float (&x)[64]) {
    float m[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) m[k] = fmaxf(x[k], x[k + 8]);
#pragma unroll
    for (int i = 16; i < 64; i += 16) {
#pragma unroll
        for (int k = 0; k < 8; ++k) m[k] = fmax3(m[k], x[i + k], x[i + k + 8]);
    }
    return fmax3(fmax3(m[0], m[1], m[2]), fmax3(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
}

// Shared-memory matrix descriptor of a 128-byte-swizzled operand: start address, leading and
// stride byte offsets (16-byte units), the descriptor version of this architecture (1 at bit
// 46) and the 128-byte swizzle mode (2 at bits 61-63).
__device__ __forceinline__ uint64_t tc_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16: fp32 accumulator, bf16 A and B, A K-major, B K-major
// (b_mn = 0) or MN-major (b_mn = 1), shape M x N.
__host__ __device__ constexpr uint32_t tc_idesc(uint32_t M, uint32_t N, uint32_t b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

// Shared memory of the tcgen05 prefill (offsets from the dynamic shared base, which the kernel
// checks to be 1024-byte aligned: no slack is reserved, so that two CTAs with three V stages
// fit one SM): the query rows [D/64][128 rows][128 B], the K stages and the V stages (a key
// block's K or V as [D/64][64 rows][128 B]), the two query blocks' key-block bitmaps, the
// barriers, the block metadata, the TMEM base and the abort flag.
struct TcSmem {
    uint32_t q, blk_bytes, kst, vst, bmA, bmB, bars, meta, taddr, abort, total;
};

__host__ __device__ inline TcSmem tc_smem_layout(int D, int nwords) {
    TcSmem s;
    uint32_t o = 0;
    s.q = o;           o += (uint32_t)kTcRows * D * 2u;
    s.blk_bytes = 64u * D * 2u;
    s.kst = o;         o += kTcKStages * s.blk_bytes;
    s.vst = o;         o += kTcVStages * s.blk_bytes;
    s.bmA = o;         o += (uint32_t)nwords * 4u;
    s.bmB = o;         o += (uint32_t)nwords * 4u;
    o = (o + 15u) & ~15u;
    s.bars = o;        o += kTcBars * 8u;
    s.meta = o;        o += kTcMetaSlots * 16u;
    s.taddr = o;       o += 16u;
    s.abort = o;       o += 16u;
    s.total = o;
    return s;
}

// The key blocks of the CTA's two query blocks, as bitmaps over blocks 0 .. qb_b: bit kb of
// bmA is set when query block qa keeps kb, of bmB when qb_b = qa + 1 keeps it (an empty bmB
// when the chunk has no query in qb_b). Both are built by all threads; a retrieval list may
// hold repeats, which the bitmap absorbs.
__device__ __forceinline__ void tc_build_bitmaps(const PfParams& p, int32_t b, int32_t kvh,
                                                 int32_t qa, bool hasB, uint32_t* bmA,
                                                 uint32_t* bmB, int32_t nw, int tid) {
    const int32_t qbb = qa + 1;
    int kind = p.head_kind ? p.head_kind[kvh] : DATTN_HEAD_DENSE;
    if (kind < 0 || kind > 2) kind = DATTN_HEAD_DENSE;
    for (int32_t w = tid; w < nw; w += kTcThreads) {
        uint32_t a = 0u, bb = 0u;
        if (kind != DATTN_HEAD_RETRIEVAL) {
            for (int bit = 0; bit < 32; ++bit) {
                const int32_t kb = 32 * w + bit;
                bool ka, kb_in;
                if (kind == DATTN_HEAD_STREAMING) {
                    ka = kb <= qa && (kb < p.sink_blocks || kb > qa - p.local_blocks);
                    kb_in = kb <= qbb && (kb < p.sink_blocks || kb > qbb - p.local_blocks);
                } else {
                    ka = kb <= qa;
                    kb_in = kb <= qbb;
                }
                a |= (ka ? 1u : 0u) << bit;
                bb |= (hasB && kb_in ? 1u : 0u) << bit;
            }
        }
        bmA[w] = a;
        bmB[w] = bb;
    }
    if (kind == DATTN_HEAD_RETRIEVAL) {
        __syncthreads();
        const int32_t* la = p.block_lists + (((int64_t)b * p.Hkv + kvh) * p.qblock_stride + qa) *
                                                p.max_sel;
        for (int32_t i = tid; i < 2 * p.max_sel; i += kTcThreads) {
            const bool second = i >= p.max_sel;
            if (second && !hasB) continue;
            const int32_t kb = __ldg(la + i);  // row qa, then row qa + 1 right after it
            const int32_t lim = second ? qbb : qa;
            if (kb >= 0 && kb <= lim)
                atomicOr(second ? bmB + (kb >> 5) : bmA + (kb >> 5), 1u << (kb & 31));
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 2)
prefill_tc_kernel(const __grid_constant__ PfParams p, const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v, int32_t nwords) {
    constexpr int KH = D / 64;  // 128-byte halves of a row
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* base = smem_raw;
    const TcSmem L = tc_smem_layout(D, nwords);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // the 128-byte swizzle of the TMA copies and the MMA operands needs 1024-byte alignment
    if ((smem_u32(base) & 1023u) != 0u) {
        if (tid == 0) set_err(p.dev_err, DATTN_DEVERR_SMEM_ALIGN);
        return;
    }
    // CTA -> (request b, group of kv_group KV heads, tile J, KV head in the group, head
    // slot): the head slots of a KV head are neighbouring CTAs, a group's tiles run together
    // with its last (longest) tiles first, and the CTAs in flight read the K/V of one group
    // only (it stays in L2). Head slot hs = KV head * spk + slot covers the query heads of
    // rows 0-63.
    const bool hp = p.head_pairs != 0;
    const int32_t spk = hp ? p.g / 2 : p.g;  // head slots per KV head
    const int32_t ngrp = p.Hkv / p.kv_group;
    int32_t c = blockIdx.x;
    const int32_t sk = c % spk;
    c /= spk;
    const int32_t hg = c % p.kv_group;
    c /= p.kv_group;
    const int32_t J = p.nqb - 1 - c % p.nqb;
    c /= p.nqb;
    const int32_t hs = ((c % ngrp) * p.kv_group + hg) * spk + sk;
    const int32_t b = c / ngrp;
    const int32_t h = hp ? 2 * hs : hs;  // the query head of rows 0-63 (rows 64-127: h + hp)
    const uint32_t bars = smem_u32(base + L.bars);
    // K and V stages are tracked apart: K_j's stage is free once S_j is computed, V_j's once
    // P_j V_j is, so the next key blocks' K loads run during this block's softmax.
    auto k_full = [&](int s) { return bars + 8u * s; };
    auto k_empty = [&](int s) { return bars + 8u * (2 + s); };
    auto v_full = [&](int s) { return bars + 8u * (4 + s); };
    auto v_empty = [&](int s) { return bars + 8u * (7 + s); };
    auto s_full = [&](int s) { return bars + 8u * (10 + s); };
    auto p_full = [&](int s) { return bars + 8u * (12 + s); };
    auto meta_full = [&](int m) { return bars + 8u * (14 + m); };
    const uint32_t pv_done = bars + 8u * 18u, drain = bars + 8u * 19u;
    int32_t* meta = reinterpret_cast<int32_t*>(base + L.meta);
    uint32_t* bmA = reinterpret_cast<uint32_t*>(base + L.bmA);
    uint32_t* bmB = reinterpret_cast<uint32_t*>(base + L.bmB);
    volatile int* abort_p = reinterpret_cast<volatile int*>(base + L.abort);
    if (tid == 0) {
        for (int s = 0; s < kTcKStages; ++s) {
            mbar_init(k_full(s), 1);
            mbar_init(k_empty(s), 1);
            mbar_init(s_full(s), 1);
            mbar_init(p_full(s), kTcSoftWarps * 32);
        }
        for (int s = 0; s < kTcVStages; ++s) {
            mbar_init(v_full(s), 1);
            mbar_init(v_empty(s), 1);
        }
        for (int m = 0; m < kTcMetaSlots; ++m) mbar_init(meta_full(m), 1);
        mbar_init(pv_done, 1);
        mbar_init(drain, 1);
        *abort_p = 0;
        fence_mbar_init();
    }
    if (warp == kTcProdWarp && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    if (warp == 0) {  // the whole warp allocates the CTA's tensor memory
        tc_alloc(smem_u32(base + L.taddr), kTcCols);
        tc_relinquish();
    }
    // V rows the MMA reads with weight 0 (tiles that are never loaded) must hold finite data:
    // zero the V stages once. Stale K needs no care: its scores are always masked, and a block
    // that skips the mask has every tile freshly loaded.
    for (uint32_t i = tid; i < kTcVStages * L.blk_bytes / 16u; i += kTcThreads)
        reinterpret_cast<uint4*>(base + L.vst)[i] = make_uint4(0u, 0u, 0u, 0u);
    tc_fence_before();
    grid_dependency_wait();  // the lengths and the pool may come from the previous kernel
    grid_launch_dependents();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = *reinterpret_cast<volatile uint32_t*>(base + L.taddr);

    // ---- the CTA's query rows and key blocks (uniform over the CTA) --------------------------
    const int32_t Ln = p.seq_lens[b];
    bool active = Ln >= p.Tq && Ln <= p.max_pages * p.P;
    if (!active && tid == 0 && hs == 0 && J == 0) set_err(p.dev_err, DATTN_DEVERR_LEN_OOB);
    const int32_t c0 = Ln - p.Tq;
    // Query block qa holds rows 0-63. Without head pairs rows 64-127 are block qa + 1 of the
    // same head; with head pairs they are block qa of head h + 1. Row r sits at position
    // qa * 64 + r (qa * 64 + r % 64 with head pairs), and the chunk's rows of the tile are the
    // positions in [p_lo, p_hi).
    const int32_t qa = (active ? c0 : 0) / kPfBlock + (hp ? J : 2 * J);
    const int32_t p_lo = max(c0, qa * kPfBlock);
    const int32_t p_hi = min(Ln, qa * kPfBlock + (hp ? kPfBlock : kTcRows));
    active = active && p_lo < p_hi;
    const bool hasB = !hp && p_hi > (qa + 1) * kPfBlock;
    const int32_t kvh = h / p.g;
    if (active && p.head_kind != nullptr && p.head_kind[kvh] == DATTN_HEAD_RETRIEVAL &&
        (qa + (hasB ? 1 : 0)) >= p.qblock_stride) {
        if (tid == 0) set_err(p.dev_err, DATTN_DEVERR_LEN_OOB);
        active = false;
    }
    const int32_t nw = active ? (qa + 1 + 1 + 31) / 32 : 0;  // words over blocks 0 .. qa + 1
    if (active) {
        tc_build_bitmaps(p, b, kvh, qa, hasB, bmA, bmB, nw, tid);
        if (hp) {  // both halves keep query block qa's key blocks
            __syncthreads();
            for (int32_t w = tid; w < nw; w += kTcThreads) bmB[w] = bmA[w];
        }
        // the query rows, in the K tiles' swizzled layout ([half][row][128 B]); with a
        // negative scale the rows are negated (exact), so that the scores scale by |scale|
        const uint32_t qneg = p.sl2 < 0.f ? 0x80008000u : 0u;
        for (int idx = tid; idx < kTcRows * (D / 8); idx += kTcThreads) {
            const int r = idx / (D / 8), ch = idx - r * (D / 8);
            const int32_t pos = qa * kPfBlock + (hp ? (r & (kPfBlock - 1)) : r);
            const int32_t hr = h + (hp && r >= kPfBlock ? 1 : 0);
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (pos >= p_lo && pos < p_hi) {
                v = __ldg(reinterpret_cast<const uint4*>(
                    p.q + (((int64_t)b * p.Tq + (pos - c0)) * p.Hq + hr) * D) + ch);
                v = make_uint4(v.x ^ qneg, v.y ^ qneg, v.z ^ qneg, v.w ^ qneg);
            }
            *reinterpret_cast<uint4*>(base + L.q + (ch >> 3) * (kTcRows * 128u) +
                                      swz128((uint32_t)r, (uint32_t)(ch & 7))) = v;
        }
        fence_proxy_async_smem();  // the tensor cores read these rows through the async proxy
    }
    __syncthreads();
    // Every role walks the same blocks in the same order: the set bits of bmA | bmB.
    int32_t nblk = 0;
    for (int32_t w = 0; w < nw; ++w) nblk += __popc(bmA[w] | bmB[w]);

    if (active && (warp == kTcProdWarp || warp == kTcVWarp)) {
        // ------------------------------------------------------ TMA producers (K, and V)
        // Both warps walk the key blocks in the same order; the K warp's ring is released by
        // S_j, the V warp's by P_j V_j, so the V copies trail the K copies by about a block.
        const bool isv = warp == kTcVWarp;
        const CUtensorMap* tmap = isv ? &tmap_v : &tmap_k;
        const uint64_t pol = policy_evict_normal();
        const uint32_t half_bytes = 64u * 128u;  // one half of a K (or V) block
        const uint32_t st0 = smem_u32(base + (isv ? L.vst : L.kst));
        const int nst = isv ? kTcVStages : kTcKStages;
        const int grp = lane >> 2, u = lane & 3;  // lane (grp, u): tile u of the group's block grp
        int32_t jk = 0;  // blocks issued
        bool ok = true;
        int32_t w = 0;
        uint32_t word = nw > 0 ? (bmA[0] | bmB[0]) : 0u;
        // the walk's next (up to) eight key blocks, one per group of four lanes; returns their
        // count and this lane's block (-1 when it has none) and flags
        auto walk = [&](int32_t& kb_o, uint32_t& fl_o) -> int {
            int n = 0;
            kb_o = -1;
            fl_o = 0u;
            for (int i = 0; i < 8; ++i) {
                while (word == 0u && ++w < nw) word = bmA[w] | bmB[w];
                if (word == 0u) break;
                const int bit = __ffs(word) - 1;
                word &= word - 1u;
                if (grp == i) {
                    kb_o = 32 * w + bit;
                    fl_o = ((bmA[w] >> bit) & 1u) | (((bmB[w] >> bit) & 1u) << 1);
                }
                ++n;
            }
            return n;
        };
        // the page of this lane's tile (read one group ahead, so its latency hides behind the
        // current group's copies)
        auto read_page = [&](int32_t kb) -> int32_t {
            const int32_t t0 = kb * kPfBlock + 16 * u;
            return kb >= 0 && t0 < p_hi ? __ldg(p.block_table + (int64_t)b * p.max_pages + t0 / p.P)
                                        : 0;
        };
        int32_t mykb;
        uint32_t myflags;
        int cnt = walk(mykb, myflags);
        int32_t page = read_page(mykb);
        while (ok && cnt > 0) {
            int32_t nkb;
            uint32_t nflags;
            const int ncnt = walk(nkb, nflags);
            const int32_t npage = read_page(nkb);
            // lane (i, u) resolves tile u of block i of this group
            int32_t y = 0, hi = 0;
            const int32_t t0 = mykb * kPfBlock + 16 * u;
            if (mykb >= 0 && t0 < p_hi) {
                if (page < 0) {
                    if (!isv) set_err(p.dev_err, DATTN_DEVERR_UNMAPPED_PAGE);
                } else if (page >= p.num_pages) {
                    if (!isv) set_err(p.dev_err, DATTN_DEVERR_PAGE_OOB);
                } else {
                    y = (page * p.Hkv + kvh) * p.P + (t0 - (t0 / p.P) * p.P);
                    hi = min(16, Ln - t0);
                }
            }
            int32_t his = hi << (5 * u), nvalid = hi > 0 ? 1 : 0;
#pragma unroll
            for (int o2 = 1; o2 < kPfTiles; o2 <<= 1) {
                his |= __shfl_xor_sync(0xffffffffu, his, o2);
                nvalid += __shfl_xor_sync(0xffffffffu, nvalid, o2);
            }
            for (int i = 0; i < cnt; ++i) {
                const int s = jk % nst, ph = (jk / nst) & 1;  // stage, and its fill's phase
                const uint32_t full = isv ? v_full(s) : k_full(s);
                if (jk >= nst && lane == 0)
                    ok = mbar_wait(isv ? v_empty(s) : k_empty(s), ph ^ 1, abort_p, p.dev_err);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                const int32_t bn = __shfl_sync(0xffffffffu, nvalid, 4 * i);
                if (!isv) {
                    const int32_t bkb = __shfl_sync(0xffffffffu, mykb, 4 * i);
                    const uint32_t bfl = __shfl_sync(0xffffffffu, myflags, 4 * i);
                    const int32_t bhis = __shfl_sync(0xffffffffu, his, 4 * i);
                    if (lane == 0) {
                        // metadata slot jk % 4 is free: block jk - 4's softmax ended before
                        // S_{jk-2} was issued, and K_jk waited for S_{jk-2}
                        int32_t* mt = meta + 4 * (jk & (kTcMetaSlots - 1));
                        mt[0] = bkb;
                        mt[1] = (int32_t)bfl;
                        mt[2] = bhis;
                        mbar_arrive(meta_full(jk & (kTcMetaSlots - 1)));
                    }
                }
                if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)bn * KH * 2048u);
                __syncwarp();
                if (grp == i && hi > 0) {
                    const uint32_t dst = st0 + (uint32_t)s * L.blk_bytes + u * 2048u;
#pragma unroll
                    for (int hh = 0; hh < KH; ++hh)
                        tma_load_3d(dst + hh * half_bytes, tmap, 0, y, hh, full, pol);
                }
                ++jk;
            }
            mykb = nkb;
            myflags = nflags;
            cnt = ncnt;
            page = npage;
        }
        // after an abort, wait (bounded in total) for copies still in flight
        if (lane == 0 && *abort_p) {
            const unsigned long long t0w = global_timer_ns();
            for (int32_t jj = max(0, jk - nst); jj < jk; ++jj)
                while (!mbar_try_wait(isv ? v_full(jj % nst) : k_full(jj % nst), (jj / nst) & 1) &&
                       global_timer_ns() - t0w < kWaitLimitNs) {
                }
        }
    } else if (active && warp == kTcMmaWarp) {
        // ---------------------------------------------------------------- MMA issuer
        if (lane == 0 && nblk > 0) {
            constexpr uint32_t idesc_s = tc_idesc(kTcRows, 64, 0);
            constexpr uint32_t idesc_o = tc_idesc(kTcRows, D, 1);
            const uint32_t qs = smem_u32(base + L.q);
            const uint32_t kst0 = smem_u32(base + L.kst), vst0 = smem_u32(base + L.vst);
            const uint32_t half_bytes = 64u * 128u;
            bool ok = true;
            // S_j = Q K_j^T into S buffer j % 2 (TMEM columns 128 + 64 (j % 2))
            auto issue_s = [&](int32_t j) {
                const int s = j & 1;
                const uint32_t kst = kst0 + (uint32_t)s * L.blk_bytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t ad =
                        tc_sdesc(qs + (kk >> 2) * (kTcRows * 128u) + (kk & 3) * 32u, 16u, 1024u);
                    const uint64_t bd = tc_sdesc(kst + (kk >> 2) * half_bytes + (kk & 3) * 32u, 16u,
                                                 1024u);
                    tc_mma_ss(tbase + 128u + 64u * s, ad, bd, idesc_s, kk > 0 ? 1u : 0u);
                }
                tc_commit(k_empty(s));
                tc_commit(s_full(s));
            };
            ok = mbar_wait(k_full(0), 0, abort_p, p.dev_err);
            if (ok) {
                tc_fence_after();
                issue_s(0);
            }
            for (int32_t j = 0; j < nblk && ok; ++j) {
                const int s = j & 1;
                if (j + 1 < nblk) {
                    ok = mbar_wait(k_full((j + 1) & 1), ((j + 1) >> 1) & 1, abort_p, p.dev_err);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(j + 1);
                }
                const int sv = j % kTcVStages;
                ok = mbar_wait(p_full(s), (j >> 1) & 1, abort_p, p.dev_err) &&
                     mbar_wait(v_full(sv), (j / kTcVStages) & 1, abort_p, p.dev_err);
                if (!ok) break;
                tc_fence_after();
                // O += P_j V_j: P from TMEM (hi terms, then lo terms), V from shared memory
                const uint32_t vst = vst0 + (uint32_t)sv * L.blk_bytes;
#pragma unroll
                for (int part = 0; part < 2; ++part) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t bd = tc_sdesc(vst + kk * 2048u, half_bytes, 1024u);
                        tc_mma_ts(tbase, tbase + 128u + 64u * s + 32u * part + 8u * kk, bd, idesc_o,
                                  (j > 0 || part > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                tc_commit(v_empty(sv));
                tc_commit(pv_done);
            }
            // every product is done: the epilogue's signal, and nothing of this CTA's may
            // still run on the tensor cores when it exits
            tc_commit(drain);
            mbar_wait(drain, 0, abort_p, p.dev_err);
        }
    } else if (active && warp < kTcSoftWarps) {
        // ---------------------------------------------------------------- softmax threads
        const int r = tid;  // this thread's query row and TMEM lane
        const int32_t pos = qa * kPfBlock + (hp ? (r & (kPfBlock - 1)) : r);
        const int32_t hr = h + (hp && r >= kPfBlock ? 1 : 0);  // this row's query head
        const bool rowok = pos >= p_lo && pos < p_hi;
        const uint32_t rbit = r >= 64 ? 2u : 1u;
        const uint32_t lanes = (uint32_t)(32 * warp) << 16;
        // |scale| log2(e) (the rows were negated for a negative scale), at least 1e-30 so that
        // a masked key (-inf) never meets a zero factor; at that floor every score is ~0
        const float sl2a = fmaxf(fabsf(p.sl2), 1e-30f);
        constexpr int32_t kFullTiles = 16 | (16 << 5) | (16 << 10) | (16 << 15);
        float m_used = kPfNegInf, m_true = kPfNegInf, l = 0.f;  // l is relative to m_used
        int32_t j = 0;
        bool ok = true;
        for (int32_t w = 0; w < nw && ok; ++w) {
            uint32_t word = bmA[w] | bmB[w];
            while (word != 0u) {
                word &= word - 1u;
                const int s = j & 1;
                // the block's metadata (slot j % 4), then its scores (s_full)
                const int ms = j & (kTcMetaSlots - 1);
                ok = mbar_wait(meta_full(ms), (j >> 2) & 1, abort_p, p.dev_err) &&
                     mbar_wait(s_full(s), (j >> 1) & 1, abort_p, p.dev_err);
                if (!__all_sync(0xffffffffu, ok)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const int32_t kb = meta[4 * ms + 0];
                const uint32_t flags = (uint32_t)meta[4 * ms + 1];
                const int32_t his = meta[4 * ms + 2];
                const uint32_t sbuf = tbase + lanes + 128u + 64u * s;
                float x[64];
                {
                    float t[32];
                    tc_ld32(sbuf, t);
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[i] = t[i];
                    tc_ld32(sbuf + 32u, t);
#pragma unroll
                    for (int i = 0; i < 32; ++i) x[32 + i] = t[i];
                    tc_wait_ld();
                }
                // mask: the row's query block keeps kb, the key is written (< length) and at
                // or before the query. Key i of tile u is kept iff i < lim[u]; a block whose
                // 64 keys all pass for every row of the warp skips the selects.
                const bool keep = rowok && (flags & rbit) != 0u;
                const int32_t cut = keep ? pos - kb * kPfBlock + 1 : 0;
                float mxr;  // the row maximum of the raw scores
                if (__all_sync(0xffffffffu, cut >= kPfBlock && his == kFullTiles)) {
                    mxr = row_max64(x);
                } else {
                    int32_t lim[kPfTiles];
#pragma unroll
                    for (int u = 0; u < kPfTiles; ++u)
                        lim[u] = min(16 * u + ((his >> (5 * u)) & 31), cut);
#pragma unroll
                    for (int i = 0; i < 64; ++i) x[i] = i < lim[i >> 4] ? x[i] : kPfNegInf;
                    mxr = row_max64(x);
                }
                const float mx = mxr * sl2a;  // scaled (log2 units); -inf stays -inf
                m_true = fmaxf(m_true, mx);
                // lazy rescale of O and l when the row maximum grows by more than 2^8; the TMEM
                // traffic is warp-collective, so a warp rescales when any of its rows must (the
                // others with factor 1)
                const bool need = mx > m_used + kTcRescale || (m_used == kPfNegInf && mx != kPfNegInf);
                const float f = need && m_used != kPfNegInf ? exp2f(m_used - mx) : 1.f;
                if (__any_sync(0xffffffffu, f != 1.f) && j > 0) {
                    // O holds the blocks before this one: wait for them, then scale it
                    mbar_wait(pv_done, (j - 1) & 1, abort_p, p.dev_err);
                    tc_fence_after();
#pragma unroll 1
                    for (int cc = 0; cc < D / 32; ++cc) {
                        float t[32];
                        tc_ld32(tbase + lanes + 32u * cc, t);
                        tc_wait_ld();
                        uint32_t u32[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) u32[i] = __float_as_uint(t[i] * f);
                        tc_st32(tbase + lanes + 32u * cc, u32);
                    }
                    tc_wait_st();
                }
                if (need) m_used = mx;
                const float mu = m_used == kPfNegInf ? 0.f : m_used;
                // p = 2^(x |scale| log2(e) - mu) in pairs (packed fp32 FMA); a masked key (-inf)
                // gives +0. P goes to the S buffer as two bf16 terms: hi (p cut to its upper 16
                // bits) into columns [0, 32), lo (the exact rest, rounded) into [32, 64).
                const uint64_t s2 = pack_f32x2(sl2a, sl2a), nmu2 = pack_f32x2(-mu, -mu);
                float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t ph[16], pl[16];
#pragma unroll
                    for (int cc = 0; cc < 16; ++cc) {
                        float p0, p1;
                        fma_f32x2(x[32 * hf + 2 * cc], x[32 * hf + 2 * cc + 1], s2, nmu2, p0, p1);
                        p0 = ex2_approx(p0);
                        p1 = ex2_approx(p1);
                        add_f32x2(ls[2 * (cc & 3)], ls[2 * (cc & 3) + 1], p0, p1);
                        const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
                        ph[cc] = __byte_perm(b0, b1, 0x7632);
                        float r0, r1;
                        sub_f32x2(p0, p1, __uint_as_float(b0 & 0xffff0000u),
                                  __uint_as_float(b1 & 0xffff0000u), r0, r1);
                        pl[cc] = pack_bf16(r0, r1);
                    }
                    tc_st16(sbuf + 16u * hf, ph);
                    tc_st16(sbuf + 32u + 16u * hf, pl);
                }
                l = l * f + (((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7])));
                tc_wait_st();
                // V rows past the length in a short tile hold stale pool data: zero them so
                // that a zero weight cannot meet a NaN
                bool short_tile = false;
#pragma unroll
                for (int u = 0; u < kPfTiles; ++u) {
                    const int32_t hi = (his >> (5 * u)) & 31;
                    short_tile = short_tile || (hi > 0 && hi < 16);
                }
                if (short_tile &&
                    mbar_wait(v_full(j % kTcVStages), (j / kTcVStages) & 1, abort_p, p.dev_err)) {
                    // (V_j's stage is refilled only after P_j V_j, which waits for this warp)
                    uint8_t* vst = base + L.vst + (uint32_t)(j % kTcVStages) * L.blk_bytes;
                    for (int idx = r; idx < kPfTiles * 16 * KH * 8; idx += kTcSoftWarps * 32) {
                        const int u = idx / (16 * KH * 8), rem = idx - u * (16 * KH * 8);
                        const int kr = rem / (KH * 8), rem2 = rem - kr * (KH * 8);
                        const int hh = rem2 >> 3, ch = rem2 & 7;
                        const int32_t hi = (his >> (5 * u)) & 31;
                        if (hi > 0 && kr >= hi)
                            *reinterpret_cast<uint4*>(vst + hh * 64u * 128u + (16 * u + kr) * 128 +
                                                      ch * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    fence_proxy_async_smem();
                }
                tc_fence_before();
                mbar_arrive(p_full(s));
                ++j;
            }
        }
        // ---- epilogue: O / l for this row (TMEM loads by the whole warp) --------------------
        // Wait for the last product on the one-phase drain barrier: pv_done may still be two
        // phases behind a warp that ran ahead of its siblings (a parity wait cannot tell those
        // phases apart).
        if (ok && nblk > 0) {
            ok = mbar_wait(drain, 0, abort_p, p.dev_err);
            tc_fence_after();
        }
        ok = __all_sync(0xffffffffu, ok);
        const int64_t row = ((int64_t)b * p.Tq + (rowok ? pos - c0 : 0)) * p.Hq + hr;
        float* orow = p.out + row * D;
        const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
        for (int cc = 0; cc < D / 32; ++cc) {
            float t[32];
            if (nblk > 0 && ok) {
                tc_ld32(tbase + lanes + 32u * cc, t);
                tc_wait_ld();
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) t[i] = 0.f;
            }
            if (rowok) {
#pragma unroll
                for (int i = 0; i < 32; i += 4)
                    *reinterpret_cast<float4*>(orow + 32 * cc + i) =
                        make_float4(t[i] * inv, t[i + 1] * inv, t[i + 2] * inv, t[i + 3] * inv);
            }
        }
        if (rowok) {
            // report the true row max and the sum relative to it
            if (p.m_out) p.m_out[row] = m_true == kPfNegInf ? kPfNegInf : m_true * kLn2;
            if (p.e_out) p.e_out[row] = m_true == kPfNegInf ? 0.f : l * exp2f(m_used - m_true);
        }
    }
    // ---- teardown: the allocating warp frees the tensor memory --------------------------------
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tc_dealloc(tbase, kTcCols);
    }
}

std::mutex g_pf_mutex;

// The pool as rows of d bf16 values split into 128-byte halves (dims {64, rows, d/64}), with
// a box of one half of 16 rows: the tcgen05 operands keep each half of a key block as 64
// contiguous 128-byte rows.
PFN_cuTensorMapEncodeTiled_v12000 tc_encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

dattn_status_t make_half_tensor_map(void* tmap_out, const void* pool, int64_t rows, int D) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = tc_encode_fn();
    if (fn == nullptr) return DATTN_ERR_CUDA;
    cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(D / 64)};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, 128};
    cuuint32_t box[3] = {64, 16, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(static_cast<CUtensorMap*>(tmap_out), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                    const_cast<void*>(pool), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? DATTN_OK : DATTN_ERR_CUDA;
}

int g_tc_smem_set[2] = {0, 0};

template <int D>
dattn_status_t launch_prefill_tc_d(const PfParams& p0, const void* k_pool, const void* v_pool,
                                   cudaStream_t stream) {
    PfParams p = p0;
    // Head pairs when a KV head has an even number of query heads: a tile is one query block
    // (a chunk touches at most ceil(Tq / 64) + 1 of them) of two heads; otherwise two query
    // blocks of one head.
    p.head_pairs = (p.g % 2 == 0) ? 1 : 0;
    const int32_t blocks = (p.Tq + kPfBlock - 1) / kPfBlock + 1;
    p.nqb = p.head_pairs ? blocks : (blocks + 1) / 2;
    const int64_t ctas = (int64_t)p.B * p.nqb * (p.head_pairs ? p.Hq / 2 : p.Hq);
    if (ctas >= (1ll << 31)) return DATTN_ERR_UNSUPPORTED;
    // The smallest group of KV heads whose tiles fill three waves of resident CTAs (two per
    // SM: each holds half the tensor memory). One KV head per group keeps the K/V in flight
    // L2-resident; a group spanning fewer waves would start a later group's long tiles so
    // late that they run alone at the end, so small chunks group all KV heads.
    {
        const int64_t per_head = (int64_t)p.nqb * (p.head_pairs ? p.g / 2 : p.g);
        const int64_t three_waves = 3ll * 2 * sm_count_current();
        p.kv_group = p.Hkv;
        for (int32_t G = 1; G < p.Hkv; ++G)
            if (p.Hkv % G == 0 && G * per_head >= three_waves) {
                p.kv_group = G;
                break;
            }
    }
    const int32_t nwords = (p.max_pages * p.P / kPfBlock + 2 + 31) / 32;
    const TcSmem L = tc_smem_layout(D, nwords);
    if (L.total > 227u * 1024u) return DATTN_ERR_UNSUPPORTED;
    {
        std::lock_guard<std::mutex> lock(g_pf_mutex);
        int& set = g_tc_smem_set[D == 128 ? 1 : 0];
        if ((int)L.total > set) {
            if (cudaFuncSetAttribute(prefill_tc_kernel<D>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)L.total) != cudaSuccess)
                return DATTN_ERR_CUDA;
            set = (int)L.total;
        }
    }
    alignas(64) CUtensorMap tk;
    alignas(64) CUtensorMap tv;
    const int64_t rows = (int64_t)p.num_pages * p.Hkv * p.P;
    dattn_status_t st;
    if ((st = make_half_tensor_map(&tk, k_pool, rows, D)) != DATTN_OK) return st;
    if ((st = make_half_tensor_map(&tv, v_pool, rows, D)) != DATTN_OK) return st;
    if (launch_pdl(prefill_tc_kernel<D>, dim3((unsigned)ctas), dim3(kTcThreads), L.total, stream,
                   p, tk, tv, nwords) != cudaSuccess)
        return DATTN_ERR_CUDA;
    return DATTN_OK;
}

bool pf_aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

}  // namespace
}  // namespace dattn

using namespace dattn;

extern "C" dattn_status_t dattn_prefill(const dattn_kv_layout* layout, const void* k_pool,
                                        const void* v_pool, const dattn_bf16* q, int32_t B,
                                        int32_t Tq, int32_t Hq, float scale,
                                        const int32_t* seq_lens,
                                        const dattn_prefill_sparse* sparse, float* out, float* m,
                                        float* e, int32_t* dev_err, void* stream) {
    // the layout checks every pool-reading call makes
    if (layout == nullptr || layout->block_table == nullptr) return DATTN_ERR_INVALID_ARG;
    if (layout->num_pages <= 0 || layout->num_kv_heads <= 0 || layout->max_pages_per_req <= 0 ||
        layout->page_size <= 0 || layout->head_dim <= 0)
        return DATTN_ERR_INVALID_ARG;
    if (layout->head_dim != 64 && layout->head_dim != 128) return DATTN_ERR_UNSUPPORTED;
    if (layout->page_size % 16 != 0 || layout->page_size > 256) return DATTN_ERR_UNSUPPORTED;
    if (layout->num_kv_heads > kMaxKvHeads) return DATTN_ERR_UNSUPPORTED;
    if ((int64_t)layout->num_pages * layout->num_kv_heads * layout->page_size >= (1ll << 31))
        return DATTN_ERR_UNSUPPORTED;
    if ((int64_t)layout->max_pages_per_req * layout->page_size >= (1ll << 30))
        return DATTN_ERR_UNSUPPORTED;
    if (layout->kv_format != DATTN_KV_BF16) {
        return layout->kv_format == DATTN_KV_FP8_E4M3 || layout->kv_format == DATTN_KV_INT4 ||
                       layout->kv_format == DATTN_KV_MIXED
                   ? DATTN_ERR_UNSUPPORTED
                   : DATTN_ERR_INVALID_ARG;
    }
    // the call's own arguments
    if (B < 0 || Tq < 0 || Hq <= 0 || Hq % layout->num_kv_heads != 0) return DATTN_ERR_INVALID_ARG;
    if (Hq / layout->num_kv_heads > kMaxGroup) return DATTN_ERR_UNSUPPORTED;
    if (B > kMaxItems) return DATTN_ERR_UNSUPPORTED;
    if (B == 0 || Tq == 0) return DATTN_OK;
    if (!k_pool || !v_pool || !q || !seq_lens || !out) return DATTN_ERR_INVALID_ARG;
    if (!pf_aligned16(k_pool) || !pf_aligned16(v_pool) || !pf_aligned16(q) || !pf_aligned16(out))
        return DATTN_ERR_INVALID_ARG;
    if ((int64_t)Tq > (int64_t)layout->max_pages_per_req * layout->page_size)
        return DATTN_ERR_INVALID_ARG;
    PfParams p{};
    if (sparse != nullptr) {
        if (!sparse->head_kind || sparse->sink_blocks < 0 || sparse->local_blocks < 0 ||
            sparse->max_sel < 0 || sparse->qblock_stride < 0)
            return DATTN_ERR_INVALID_ARG;
        if (sparse->max_sel > 0 && (!sparse->block_lists || sparse->qblock_stride == 0))
            return DATTN_ERR_INVALID_ARG;
        if ((int64_t)B * layout->num_kv_heads * sparse->qblock_stride * sparse->max_sel >=
            (1ll << 31))
            return DATTN_ERR_UNSUPPORTED;
        p.head_kind = sparse->head_kind;
        p.sink_blocks = sparse->sink_blocks;
        p.local_blocks = sparse->local_blocks;
        p.max_sel = sparse->max_sel;
        p.qblock_stride = sparse->qblock_stride;
        p.block_lists = sparse->block_lists;
    }
    p.num_pages = layout->num_pages;
    p.Hkv = layout->num_kv_heads;
    p.P = layout->page_size;
    p.max_pages = layout->max_pages_per_req;
    p.block_table = layout->block_table;
    p.q = q;
    p.B = B;
    p.Tq = Tq;
    p.Hq = Hq;
    p.g = Hq / p.Hkv;
    p.sl2 = scale * kLog2e;
    p.seq_lens = seq_lens;
    p.nqb = (Tq + kPfBlock - 1) / kPfBlock + 1;  // a chunk spans at most this many blocks
    p.out = out;
    p.m_out = m;
    p.e_out = e;
    p.dev_err = dev_err;
    const int64_t ctas = (int64_t)B * p.nqb * Hq;
    if (ctas >= (1ll << 31)) return DATTN_ERR_UNSUPPORTED;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return layout->head_dim == 64 ? launch_prefill_tc_d<64>(p, k_pool, v_pool, s)
                                  : launch_prefill_tc_d<128>(p, k_pool, v_pool, s);
}
