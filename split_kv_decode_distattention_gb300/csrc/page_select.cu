// Page scoring and top-K page selection for retrieval heads (dattn_page_select).
//
// "LLM长序列服务优化：LServe的块稀疏注意力技术":
//   §2.2.2 (解码阶段创新): a 64-token physical page holds four 16-token logical pages, each
//     with per-channel k_max / k_min. Pages are scored against the query, and the
//     selection is made once at the start of a window of decode steps, then reused.
//   §3.1.2 (动态稀疏的层次化选择): the physical-page score is the max over its logical
//     pages, and the K highest-scoring physical pages are kept.
// The logical score is sum_d max(q_d * kmax_d, q_d * kmin_d), an upper bound of q . k for
// every key of the logical page. With g query heads per KV head, the score is the max over
// the g heads, so one selection serves the whole group.
//
// GB300 design. The statistics scan is HBM-bound: every reuse window it reads all k_max and
// k_min of the retrieval heads (512 B per logical page at d = 128), and it must score them
// at that speed. The physical pages of all retrieval (request, KV head) pairs are laid end
// to end and cut into equal contiguous ranges, one per CTA.
//  - Scoring is a dense contraction: for a unit of 16 logical pages the scores of the g
//    query heads are [k_max | k_min] (16 x 2d, bf16) times [max(q,0) | min(q,0)]^T (2d x g,
//    bf16), which runs on the tensor cores (mma m16n8k16, the 16 pages on M, the heads on N).
//    One of max(q,0), min(q,0) is an exact zero per channel, so the contraction adds exactly
//    the products the score definition picks, and every product of two bf16 values is exact.
//  - A unit's physical pages arrive by one bulk copy each (up to 2 KB at P = 64), staged so
//    that the ldmatrix reads of the 16-row tile meet at most 2-way bank conflicts (see
//    sel_stage_bytes). Sixteen warps per SM keep enough copies in flight; each holds as many
//    units as shared memory allows and refills a stage as soon as it has read it. Units
//    (whole physical pages) are handed to the warps by a shared counter, so faster warps take
//    more. Block-table entries of a piece are staged in shared memory first.
//  - Rounding: each 16-channel k-step runs with a zero accumulator and its result is added
//    to the running sum in fp32 (round to nearest), in a fixed order. Whatever rounding the
//    tensor core applies inside one k-step (16 exact products), the sum stays far inside the
//    bound the selection is held to for any fp32 evaluation, d * 2^-23 * sum |terms|.
//  - The physical-page score is a max over adjacent lanes (heads, then logical pages). Page
//    maxima that reach the running K-th key go to a per-warp candidate buffer, folded into
//    the warp's top K by a warp-synchronous bitonic sort.
//  - At the end of a piece the warps' lists are merged. A head split across CTAs leaves each
//    CTA's top K in the workspace, and the CTA that arrives last merges them.
#include "common.cuh"
#include "internal.h"

namespace dattn {

namespace {

// Warps per CTA (one CTA per SM): sixteen keep enough bulk copies in flight per SM. The
// warps' lists are merged pairwise, so the count is a power of two.
constexpr int kSelWarps = 16;
constexpr int kSelMaxWarps = kSelWarps;
static_assert((kSelWarps & (kSelWarps - 1)) == 0, "pairwise list merges need 2^n warps");

struct SelParams {
    int32_t num_pages, Hkv, P, max_pages;
    const int32_t* block_table;
    const uint16_t* stats;
    const uint16_t* q;
    int32_t B, Hq, g;
    const int32_t* seq_lens;
    const int8_t* head_kind;
    int32_t top_k;
    int32_t* selected;
    int32_t* selected_phys;  // nullable: the pool page of each selected page
    int32_t* counters;
    uint64_t* slots;
    int32_t nseg;
    int32_t stages;  // units of statistics rows staged per warp
    int32_t* dev_err;
};

__host__ __device__ inline int next_pow2(int x) {
    int n = 1;
    while (n < x) n <<= 1;
    return n;
}

// Block-table entries staged in shared memory at once. A CTA's range of one head is restaged
// (its copies drained first) every kSelBT pages; 4096 covers the range of a CTA at the
// sizes measured (1724 pages per CTA at 512K tokens, batch 8): 1024 took 115.4 µs, 4096
// 112.9 µs.
constexpr int kSelBT = 4096;
// Units of fixed cost per retrieval (request, KV head) in the split: the query fetch, the
// block-table staging and pipeline fill, and the lists' merge and hand-off of a piece. The
// split cuts pages plus these units evenly, so a CTA whose range starts a head takes fewer
// pages. Measured at 512K tokens, batch 8 (1724 pages per CTA): 0 units 112.6 µs, 64 110.6,
// 160 108.3, 256 104.5, 384 and 512 106.5.
constexpr int kSelSegCost = 256;

struct SelSmem {
    uint32_t flags, stage, bars, masks, batches, bt, wbuf, ret_before, ret_heads, item_start,
        item_len, scan, total;
    int kp, wn, stages;
};

// nw: warps per CTA; stage_bytes: one unit of statistics rows; stages: units staged per
// warp.
__host__ __device__ inline SelSmem sel_smem_layout(int B, int Hkv, int K, int nw,
                                                   uint32_t stage_bytes, int stages) {
    SelSmem s;
    s.stages = stages;
    s.kp = next_pow2(K);                     // list length: K rounded up to a power of two
    // per-warp buffer: running list, then room for max(Kp, 32) candidates (a power of two;
    // a unit adds up to 16 before a fold)
    s.wn = s.kp + (s.kp > 32 ? s.kp : 32);
    uint32_t o = 0;
    // +0: last-arrival flag, +4: abort flag, +8: next unit, +16: CTA-wide K-th key
    s.flags = o;      o += 32u;
    o = (o + 127u) & ~127u;
    s.stage = o;      o += (uint32_t)(nw * stages) * stage_bytes;
    s.bars = o;       o += (uint32_t)(nw * stages) * 8u;
    s.masks = o;      o += (uint32_t)(nw * stages) * 4u;
    s.batches = o;    o += (uint32_t)(nw * stages) * 4u;
    s.bt = o;         o += kSelBT * 4u;
    s.wbuf = o;       o += (uint32_t)nw * s.wn * 8u;
    s.ret_before = o; o += (uint32_t)(Hkv + 1) * 4u;
    s.ret_heads = o;  o += (uint32_t)Hkv * 4u;
    o = (o + 15u) & ~15u;
    s.item_start = o; o += (uint32_t)(B + 1) * 4u;
    s.item_len = o;   o += (uint32_t)B * 4u;
    o = (o + 15u) & ~15u;
    s.scan = o;       o += (uint32_t)kSelMaxWarps * 4u;
    s.total = o + 128u;
    return s;
}

__device__ __forceinline__ uint64_t make_key(float score, int32_t page) {
    const uint32_t u = __float_as_uint(score + 0.0f);  // -0 becomes +0
    const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((uint64_t)ord << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)page);
}

// Score of a key from make_key (-inf for the empty key 0).
__device__ __forceinline__ float key_score(uint64_t key) {
    if (key == 0ull) return -__int_as_float(0x7f800000);
    const uint32_t ord = (uint32_t)(key >> 32);
    return __uint_as_float((ord & 0x80000000u) ? (ord & 0x7fffffffu) : ~ord);
}

// Bitonic sort of buf[0..n) into descending order by nthreads threads (index tid); sync()
// separates the steps.
template <typename Sync>
__device__ __forceinline__ void bitonic_desc(uint64_t* buf, int n, int tid, int nthreads,
                                             Sync sync) {
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int idx = tid; idx < (n >> 1); idx += nthreads) {
                const int i = ((idx & ~(j - 1)) << 1) | (idx & (j - 1));  // j is a power of 2
                const int l = i + j;
                const uint64_t x = buf[i], y = buf[l];
                const bool desc = (i & k) == 0;
                if (desc ? (x < y) : (x > y)) {
                    buf[i] = y;
                    buf[l] = x;
                }
            }
            sync();
        }
    }
}

// Warp-synchronous merge of two descending lists a[0..n) and b[0..n) (n a power of two):
// a becomes the n largest keys of both, descending. c[i] = max(a[i], b[n-1-i]) holds those
// keys as a bitonic sequence, which a cascade of half-cleaners sorts.
__device__ __forceinline__ void warp_merge_desc(uint64_t* a, const uint64_t* b, int n, int lane) {
    for (int i = lane; i < n; i += 32) {
        const uint64_t x = a[i], y = b[n - 1 - i];
        a[i] = x > y ? x : y;
    }
    __syncwarp();
    for (int j = n >> 1; j > 0; j >>= 1) {
        for (int idx = lane; idx < (n >> 1); idx += 32) {
            const int i = ((idx & ~(j - 1)) << 1) | (idx & (j - 1));
            const uint64_t x = a[i], y = a[i + j];
            if (x < y) {
                a[i] = y;
                a[i + j] = x;
            }
        }
        __syncwarp();
    }
}


// The logical pages of one unit (the mma's M).
constexpr int kUnitRows = 16;

// Staging of a unit. With up to 4 logical pages per physical page, a physical page's rows
// arrive by one bulk copy at a stride of LPG rows plus 16 bytes, and row i of the unit's mma
// tile is logical page i / UPP of physical page i % UPP: the eight rows an ldmatrix reads
// then come from at least two physical pages each in a distinct bank group (a 2-way
// conflict at most). With 8 or 16 logical pages per physical page, every logical page has
// its own copy and row stride 2d bf16 plus 16 bytes (no conflict).
__host__ __device__ constexpr bool sel_page_copies(int LPG) { return LPG <= 4; }
__host__ __device__ constexpr uint32_t sel_stage_bytes(int D, int LPG) {
    return sel_page_copies(LPG) ? (uint32_t)(16 / LPG) * ((uint32_t)LPG * 4u * D + 16u)
                                : 16u * (4u * (uint32_t)D + 16u);
}

// d = a * b with a zero accumulator (m16n8k16, bf16 in, fp32 out).
__device__ __forceinline__ void mma_bf16_zero_acc(float (&d)[4], uint32_t a0, uint32_t a1,
                                                  uint32_t a2, uint32_t a3, uint32_t b0,
                                                  uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// The positive part max(x, 0) and the negative part min(x, 0) of two bf16 values, exactly
// (a value keeps its bits or becomes +0).
__device__ __forceinline__ uint32_t bf16x2_pos(uint32_t w) {
    const uint32_t neg = ((w >> 15) & 0x00010001u) * 0xffffu;
    return w & ~neg;
}
__device__ __forceinline__ uint32_t bf16x2_neg(uint32_t w) {
    const uint32_t neg = ((w >> 15) & 0x00010001u) * 0xffffu;
    return w & neg;
}

// Adds bytes to the transaction count of the barrier's current phase (no arrival).
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// D: head_dim; LPG: logical pages per physical page (P / 16, a power of two).
template <int D, int LPG>
__global__ void __launch_bounds__(kSelWarps * 32, 1)
page_select_kernel(const __grid_constant__ SelParams p) {
    constexpr int NW = kSelWarps;
    constexpr int NT = NW * 32;
    constexpr int KS = 2 * D / 16;             // k-steps over the 2d channels [k_max | k_min]
    constexpr int UPP = kUnitRows / LPG;       // physical pages per unit
    constexpr uint32_t kRowBytes = 4u * D;     // one logical page's row: k_max and k_min
    constexpr bool kPageCopies = sel_page_copies(LPG);
    // byte offset of a physical page and of a row within it in a stage
    constexpr uint32_t kPageStride = kPageCopies ? LPG * kRowBytes + 16u : LPG * (kRowBytes + 16u);
    constexpr uint32_t kRowStride = kPageCopies ? kRowBytes : kRowBytes + 16u;
    constexpr uint32_t kStageBytes = sel_stage_bytes(D, LPG);
    static_assert(kStageBytes >= UPP * kPageStride, "stage holds the unit");
    const float kNInf = -__int_as_float(0x7f800000);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_off = smem_u32(smem_raw);
    uint8_t* base = smem_raw + (((raw_off + 127u) & ~127u) - raw_off);
    const int K = p.top_k;
    const SelSmem L = sel_smem_layout(p.B, p.Hkv, K, NW, kStageBytes, p.stages);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t G = gridDim.x, cta = blockIdx.x;
    int* last_flag = reinterpret_cast<int*>(base + L.flags);
    int32_t* ret_before = reinterpret_cast<int32_t*>(base + L.ret_before);
    int32_t* ret_heads = reinterpret_cast<int32_t*>(base + L.ret_heads);
    int32_t* item_start = reinterpret_cast<int32_t*>(base + L.item_start);
    int32_t* item_len = reinterpret_cast<int32_t*>(base + L.item_len);
    int32_t* scan = reinterpret_cast<int32_t*>(base + L.scan);

    if (tid == 0) reinterpret_cast<volatile int*>(base + L.flags)[1] = 0;  // abort flag
    {  // warm L2 with the metadata read right after the wait (each line by one thread)
        const int64_t gt = (int64_t)cta * NT + tid, gn = (int64_t)G * NT;
        prefetch_l2_range(p.seq_lens, (size_t)p.B * 4u, gt, gn);
        const size_t bt_bytes = (size_t)p.B * p.max_pages * 4u;
        if (bt_bytes <= (16u << 20)) prefetch_l2_range(p.block_table, bt_bytes, gt, gn);
        prefetch_l2_range(p.q, (size_t)p.B * p.Hq * D * 2u, gt, gn);
    }
    grid_dependency_wait();  // lengths and statistics may come from the previous kernel
    grid_launch_dependents();
    // ---------------------------------------------------------------- setup
    for (int h = tid; h < p.Hkv; h += NT)
        ret_heads[h] = p.head_kind[h] == DATTN_HEAD_RETRIEVAL ? 1 : 0;
    __syncthreads();
    if (tid == 0) {
        int32_t r = 0;
        for (int h = 0; h < p.Hkv; ++h) {
            const int isr = ret_heads[h];
            ret_before[h] = r;
            if (isr) ret_heads[r++] = h;  // compacts in place: r <= h
        }
        ret_before[p.Hkv] = r;
    }
    __syncthreads();
    const int32_t nret = ret_before[p.Hkv];
    {
        const int32_t n = p.B;
        const int32_t per = (n + NT - 1) / NT;
        const int32_t i0 = min(n, tid * per), i1 = min(n, i0 + per);
        int32_t local_sum = 0;
        for (int32_t i = i0; i < i1; ++i) {
            int32_t Lb = p.seq_lens[i];
            const int32_t cap = p.max_pages * p.P;
            if (Lb < 0 || Lb > cap) {
                set_err(p.dev_err, DATTN_DEVERR_LEN_OOB);
                Lb = min(max(Lb, 0), cap);
            }
            item_len[i] = Lb;
            const int32_t np = (Lb + p.P - 1) / p.P;
            const int32_t cnt = nret * (np > 0 ? np + kSelSegCost : 0);
            item_start[i] = cnt;
            local_sum += cnt;
        }
        int32_t incl = local_sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        if (lane == 31) scan[warp] = incl;
        __syncthreads();
        int32_t run = incl - local_sum;
        for (int w = 0; w < warp; ++w) run += scan[w];
        for (int32_t i = i0; i < i1; ++i) {
            const int32_t c = item_start[i];
            item_start[i] = run;
            run += c;
        }
        if (tid == 0) {
            int32_t tot = 0;
            for (int w = 0; w < NW; ++w) tot += scan[w];
            item_start[n] = tot;
        }
        __syncthreads();
    }
    const int32_t W = item_start[p.B];
    auto npages_of = [&](int32_t b) { return (item_len[b] + p.P - 1) / p.P; };
    // A retrieval segment of n > 0 pages spans n + kSelSegCost positions of the split: its
    // fixed cost, then its pages. st: the span's first position; len: n (0 for other heads).
    auto seg_span = [&](int32_t s, int32_t& st, int32_t& len) {
        const int32_t b = s / p.Hkv, h = s - b * p.Hkv;
        const int32_t n = npages_of(b);
        const bool ret = p.head_kind[h] == DATTN_HEAD_RETRIEVAL;
        st = item_start[b] + ret_before[h] * (n > 0 ? n + kSelSegCost : 0);
        len = ret ? n : 0;
    };
    auto locate = [&](int32_t t) {  // segment whose span holds position t
        int32_t lo = 0, hi = p.B - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (item_start[mid] <= t) lo = mid; else hi = mid - 1;
        }
        const int32_t n = npages_of(lo);
        const int32_t r = (t - item_start[lo]) / (n + kSelSegCost);
        return lo * p.Hkv + ret_heads[r];
    };
    // only the first min(G, W) CTAs take units, so each participating CTA owns at least one
    const int32_t Gw = W < G ? (W > 0 ? W : 1) : G;
    const int32_t t_begin = cta < Gw ? (int32_t)split_begin(W, Gw, cta) : 0;
    const int32_t t_end = cta < Gw ? (int32_t)split_begin(W, Gw, cta + 1) : 0;

    // rows of heads without units (other kinds, or empty requests) are all -1
    for (int32_t s = cta; s < p.nseg; s += G) {
        int32_t st, len;
        seg_span(s, st, len);
        if (len == 0)
            for (int r = tid; r < K; r += NT) {
                p.selected[(int64_t)s * K + r] = -1;
                if (p.selected_phys) p.selected_phys[(int64_t)s * K + r] = -1;
            }
    }
    if (t_begin >= t_end) return;

    const int Kp = L.kp;  // K rounded up to a power of two; key 0 marks an empty entry
    uint64_t* wbuf_all = reinterpret_cast<uint64_t*>(base + L.wbuf);
    uint64_t* wbuf = wbuf_all + warp * L.wn;  // [0, Kp): running top keys; then candidates
    const int capw = L.wn - Kp;
    auto csync = [&]() { __syncthreads(); };
    auto wsync = [&]() { __syncwarp(); };
    // Folds the candidates wbuf[Kp .. Kp+cnt) into the running list wbuf[0 .. Kp): sorts
    // the candidates (padded to a power of two), then merges their top Kp into the list.
    auto warp_fold = [&](int cnt) {
        const int m = next_pow2(cnt);
        const int top = m > Kp ? m : Kp;
        for (int i = Kp + cnt + lane; i < Kp + top; i += 32) wbuf[i] = 0ull;
        __syncwarp();
        bitonic_desc(wbuf + Kp, m, lane, 32, wsync);
        warp_merge_desc(wbuf, wbuf + Kp, Kp, lane);
    };
    // the list of warp w after the pieces' and warps' lists are merged: sorted descending
    auto list_of = [&](int w) { return wbuf_all + w * L.wn; };
    // merges the warps' running lists into list_of(0) (log2(NW) levels of pairwise merges)
    auto merge_warps = [&]() {
#pragma unroll 1
        for (int n = NW / 2; n >= 1; n >>= 1) {
            if (warp < n) warp_merge_desc(list_of(warp), list_of(warp + n), Kp, lane);
            csync();
        }
    };
    // list_of(0)[0 .. K): top K keys -> selected row of segment seg, ascending pages
    auto finalize = [&](int32_t seg) {
        if (warp == 0) {
            uint64_t* f = list_of(0);
            for (int i = lane; i < Kp; i += 32)
                f[i] = (i < K && f[i] != 0ull) ? (f[i] & 0xFFFFFFFFull) : 0ull;
            __syncwarp();
            bitonic_desc(f, Kp, lane, 32, wsync);  // low word descending = page ascending
            const int32_t* btrow = p.block_table + (int64_t)(seg / p.Hkv) * p.max_pages;
            for (int r = lane; r < K; r += 32) {
                const uint64_t kk = f[r];
                const int32_t pg = kk ? (int32_t)(0xFFFFFFFFu - (uint32_t)kk) : -1;
                p.selected[(int64_t)seg * K + r] = pg;
                if (p.selected_phys) p.selected_phys[(int64_t)seg * K + r] = pg >= 0 ? btrow[pg] : -1;
            }
        }
        csync();
    };

    const uint64_t pol = policy_evict_first();
    int32_t* bt_s = reinterpret_cast<int32_t*>(base + L.bt);
    const int g8 = lane >> 2, tig = lane & 3;
    // ldmatrix lane address within a unit: tile row i = (lane & 7) + 8 ((lane >> 3) & 1),
    // 16-byte chunk lane >> 4 of the k-step's 32 bytes. Row i is logical page (i / UPP) of
    // physical page (i % UPP) with page copies, else logical page (i % LPG) of physical page
    // (i / LPG).
    const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8;
    const uint32_t lrow_off =
        (kPageCopies ? (uint32_t)(lrow % UPP) * kPageStride + (uint32_t)(lrow / UPP) * kRowStride
                     : (uint32_t)(lrow / LPG) * kPageStride + (uint32_t)(lrow % LPG) * kRowStride) +
        (uint32_t)(lane >> 4) * 16u;
    // This warp's stages: S units of 16 padded rows each, filled by bulk copies.
    const int S = L.stages;
    const uint32_t stage0 = smem_u32(base + L.stage) + (uint32_t)(warp * S) * kStageBytes;
    const uint32_t bar0 = smem_u32(base + L.bars) + (uint32_t)(warp * S) * 8u;
    uint32_t* smask = reinterpret_cast<uint32_t*>(base + L.masks) + warp * S;
    int32_t* sunit = reinterpret_cast<int32_t*>(base + L.batches) + warp * S;
    int32_t* next_unit = reinterpret_cast<int32_t*>(base + L.flags + 8);
    unsigned long long* cta_thresh_u = reinterpret_cast<unsigned long long*>(base + L.flags + 16);
    volatile uint64_t* cta_thresh = reinterpret_cast<volatile uint64_t*>(cta_thresh_u);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L.flags + 4);
    if (lane < S) mbar_init(bar0 + 8u * lane, 1);
    fence_mbar_init();
    __syncwarp();
    // The warp uses its stages round robin over the whole kernel. (st, par) is the stage of
    // the next unit to wait for and the parity of the phase that unit completes; every unit
    // issued is eventually waited for or skipped with advance().
    int st = 0;
    uint32_t par = 0u;
    auto advance = [&]() {
        if (++st == S) {
            st = 0;
            par ^= 1u;
        }
    };

    int32_t apos = t_begin;  // position in the split
    int32_t s = locate(t_begin);
    while (apos < t_end && !*abort_flag) {
        int32_t sst0, slen;
        seg_span(s, sst0, slen);
        while (slen == 0 || sst0 + kSelSegCost + slen <= apos) {
            if (++s >= p.nseg) break;
            seg_span(s, sst0, slen);
        }
        if (s >= p.nseg) break;
        // the piece: the segment's pages within [apos, t_end), in page positions a .. pe of the
        // segment's own pages sst .. sst + slen
        const int32_t sst = sst0 + kSelSegCost;
        const int32_t a = max(apos, sst), pe = min(sst + slen, t_end);
        if (a >= pe) break;  // the range ends within the segment's fixed cost
        const int32_t b = s / p.Hkv, h = s - b * p.Hkv;
        const int32_t Lb = item_len[b];
        // B fragments of [max(q,0) | min(q,0)]^T: lane holds column (query head) g8 at the
        // k-step's channel pairs 2 tig, 2 tig + 1 and 2 tig + 8, 2 tig + 9 (heads >= g are 0)
        uint32_t bq[KS][2];
        {
            const bool ok = g8 < p.g;
            const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
                p.q + ((int64_t)b * p.Hq + h * p.g + (ok ? g8 : 0)) * D);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const int c = (16 * ks) % D;  // channel of the k-step within q
                const uint32_t w0 = ok ? __ldg(qrow + c / 2 + tig) : 0u;
                const uint32_t w1 = ok ? __ldg(qrow + c / 2 + 4 + tig) : 0u;
                const bool posp = 16 * ks < D;  // k_max half: max(q,0); k_min half: min(q,0)
                bq[ks][0] = posp ? bf16x2_pos(w0) : bf16x2_neg(w0);
                bq[ks][1] = posp ? bf16x2_pos(w1) : bf16x2_neg(w1);
            }
        }
        for (int i = lane; i < L.wn; i += 32) wbuf[i] = 0ull;
        int cnt_c = 0;
        uint64_t thresh = 0ull;  // running K-th key of the warp (0 while fewer than K)
        float thr_sc = kNInf;    // its score
        const int32_t* btrow = p.block_table + (int64_t)b * p.max_pages;
        const int32_t pr0 = a - sst;  // first page of the piece (request-relative)
        for (int32_t cb = 0; cb < pe - a && !*abort_flag; cb += kSelBT) {
            const int32_t nc = min(kSelBT, pe - a - cb);  // pages of this block
            const int32_t pg0 = pr0 + cb;                 // request-relative page of bt_s[0]
            for (int i = tid; i < nc; i += NT) bt_s[i] = btrow[pg0 + i];
            if (tid == 0) {
                *next_unit = 0;
                if (cb == 0) *cta_thresh = 0ull;
            }
            csync();
            const int32_t nunits = (nc + UPP - 1) / UPP;
            // Issues the next unit of this warp into stage st, or marks the stage empty (-1)
            // once the units are exhausted. With page copies lane t < UPP takes physical page
            // t of the unit: its logical pages that hold tokens are a prefix of nv rows,
            // copied at once. Otherwise lane r < 16 takes logical page r % LPG of physical
            // page r / LPG. smask[st] gets the mask of tile rows copied; the others are never
            // scored.
            auto issue = [&](int st) {
                int32_t u = 0;
                if (lane == 0) u = atomicAdd(next_unit, 1);
                u = __shfl_sync(0xffffffffu, u, 0);
                const int32_t bi = u < nunits ? u : -1;
                const uint32_t bar = bar0 + 8u * st;
                constexpr int kLanes = kPageCopies ? UPP : kUnitRows;
                int32_t nv = 0, phys = -1, t = 0, lp = 0;
                if (bi >= 0 && lane < kLanes) {
                    t = kPageCopies ? lane : lane / LPG;
                    lp = kPageCopies ? 0 : lane % LPG;
                    const int32_t pc = bi * UPP + t;
                    if (pc < nc) {
                        const int32_t rem = Lb - (pg0 + pc) * p.P - lp * 16;
                        nv = min(max((rem + 15) >> 4, 0), kPageCopies ? LPG : 1);
                        phys = bt_s[pc];
                        if (nv > 0 && (phys < 0 || phys >= p.num_pages)) {
                            if (lp == 0)
                                set_err(p.dev_err, phys < 0 ? DATTN_DEVERR_UNMAPPED_PAGE
                                                            : DATTN_DEVERR_PAGE_OOB);
                            nv = 0;
                        }
                    }
                }
                // tile rows copied: with page copies rows t + UPP lp for lp < nv, else row lane
                uint32_t part = 0u;
                if (kPageCopies) {
                    for (int l = 0; l < nv; ++l) part |= 1u << (t + UPP * l);
                } else if (nv > 0) {
                    part = 1u << lane;
                }
                const uint32_t mask = __reduce_or_sync(0xffffffffu, part);
                const uint32_t bytes = (uint32_t)nv * kRowBytes;
                if (bytes) mbar_expect_tx(bar, bytes);
                __syncwarp();
                if (lane == 0) {
                    smask[st] = mask;
                    sunit[st] = bi;
                    mbar_arrive(bar);
                }
                if (bytes) {
                    const uint16_t* src =
                        p.stats + (((int64_t)phys * p.Hkv + h) * LPG + lp) * (2 * D);
                    bulk_copy(stage0 + (uint32_t)st * kStageBytes + (uint32_t)t * kPageStride +
                                  (uint32_t)lp * kRowStride,
                              src, bytes, bar, pol);
                }
            };
            for (int k = 0, t = st; k < S; ++k, t = (t + 1 == S) ? 0 : t + 1) issue(t);
            int32_t pending = S;  // units issued and not yet waited for
            // Offers the score sc of physical page pc (block-relative) held by this lane when
            // own: keys are built only when some page reaches the K-th score so far (the
            // larger of the warp's and the CTA's); ties are settled by the full key.
            auto offer = [&](bool own, int32_t pc, float sc) {
                const uint64_t th = max(thresh, *cta_thresh);
                const float th_sc = th == thresh ? thr_sc : key_score(th);
                const bool cand = own && sc != kNInf && sc >= th_sc;
                if (__any_sync(0xffffffffu, cand)) {
                    const uint64_t key = cand ? make_key(sc, pg0 + pc) : 0ull;
                    const bool take = key > th;
                    const uint32_t bal = __ballot_sync(0xffffffffu, take);
                    if (take) wbuf[Kp + cnt_c + __popc(bal & ((1u << lane) - 1u))] = key;
                    cnt_c += __popc(bal);
                    __syncwarp();
                    if (cnt_c > capw - 32) {
                        warp_fold(cnt_c);
                        cnt_c = 0;
                        thresh = wbuf[K - 1];
                        thr_sc = key_score(thresh);
                        if (lane == 0 && thresh) atomicMax(cta_thresh_u, thresh);
                    }
                }
            };
            while (true) {
                // warp-uniform, bounded wait for the stage's copies
                const bool ok = __all_sync(0xffffffffu,
                                           mbar_wait(bar0 + 8u * st, par, abort_flag, p.dev_err));
                if (!ok) break;
                const int cst = st;
                advance();
                --pending;
                const int32_t bi = sunit[cst];
                if (bi < 0) break;  // the units are exhausted; later stages are empty too
                const uint32_t mask = smask[cst];
                // scores of the unit's 16 logical pages (rows) for the 8 query-head columns:
                // one zero-accumulator mma per 16-channel k-step, summed in fp32 in k order
                const uint32_t sbase = stage0 + (uint32_t)cst * kStageBytes + lrow_off;
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(sbase + (uint32_t)ks * 32u, a0, a1, a2, a3);
                    float t[4];
                    mma_bf16_zero_acc(t, a0, a1, a2, a3, bq[ks][0], bq[ks][1]);
                    acc[0] += t[0];
                    acc[1] += t[1];
                    acc[2] += t[2];
                    acc[3] += t[3];
                }
                // every lane has read the stage: refill it with the warp's next unit
                __syncwarp();
                fence_proxy_async_smem();
                issue(cst);
                ++pending;
                // lane: tile rows g8 and g8 + 8, heads 2 tig and 2 tig + 1; max over the g
                // heads, then over the logical pages of each physical page
                const bool h0 = 2 * tig < p.g, h1 = 2 * tig + 1 < p.g;
                float vlo = ((mask >> g8) & 1u) ? fmaxf(h0 ? acc[0] : kNInf, h1 ? acc[1] : kNInf)
                                                : kNInf;
                float vhi = ((mask >> (g8 + 8)) & 1u)
                                ? fmaxf(h0 ? acc[2] : kNInf, h1 ? acc[3] : kNInf)
                                : kNInf;
#pragma unroll
                for (int o = 1; o < 4; o <<= 1) {
                    vlo = fmaxf(vlo, __shfl_xor_sync(0xffffffffu, vlo, o));
                    vhi = fmaxf(vhi, __shfl_xor_sync(0xffffffffu, vhi, o));
                }
                if constexpr (LPG == 1) {
                    // rows g8 and g8 + 8 are physical pages g8 and g8 + 8
                    offer(tig == 0, bi * UPP + g8, vlo);
                    offer(tig == 0, bi * UPP + g8 + 8, vhi);
                } else if constexpr (kPageCopies) {
                    // rows g8 and g8 + 8 are logical pages of physical page g8 % UPP; the
                    // lanes g8 + UPP m hold its other logical pages
                    float v = fmaxf(vlo, vhi);
#pragma unroll
                    for (int o = 4 * UPP; o < 32; o <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                    offer(tig == 0 && g8 < UPP, bi * UPP + g8, v);
                } else {
                    // rows g8 and g8 + 8 are logical pages of physical pages g8 / LPG and
                    // (g8 + 8) / LPG
#pragma unroll
                    for (int o = 4; o < 4 * 8; o <<= 1) {
                        vlo = fmaxf(vlo, __shfl_xor_sync(0xffffffffu, vlo, o));
                        vhi = fmaxf(vhi, __shfl_xor_sync(0xffffffffu, vhi, o));
                    }
                    if constexpr (LPG == 16) {
                        offer(lane == 0, bi * UPP, fmaxf(vlo, vhi));
                    } else {
                        offer(lane == 0, bi * UPP, vlo);
                        offer(lane == 0, bi * UPP + 1, vhi);
                    }
                }
            }
            // Step over the units issued and not waited for. After a normal end they are
            // empty stages (no copies, their phases complete at once); after an abort, wait
            // (bounded) for the copies still in flight.
            for (; pending > 0; --pending) {
                if (*abort_flag) {
                    const unsigned long long t0 = global_timer_ns();
                    while (!mbar_try_wait(bar0 + 8u * st, par) &&
                           global_timer_ns() - t0 < kWaitLimitNs) {
                    }
                }
                advance();
            }
            csync();  // bt_s is restaged for the next block of pages
        }
        if (cnt_c > 0) warp_fold(cnt_c);
        csync();
        merge_warps();
        const bool whole = (a == sst) && (pe == sst + slen);
        if (whole) {
            finalize(s);
        } else {
            uint64_t* my = p.slots + (int64_t)(cta + s) * K;
            for (int r = tid; r < K; r += NT) my[r] = list_of(0)[r];
            csync();
            const int32_t c_first = split_owner(sst, W, Gw);
            const int32_t c_last = split_owner(sst + slen - 1, W, Gw);
            const int32_t npieces = c_last - c_first + 1;
            if (tid == 0) {
                // release this CTA's list, acquire the others' if this is the last piece
                const int32_t prev = atom_add_acq_rel_gpu(p.counters + s, 1);
                *last_flag = (prev == npieces - 1) ? 1 : 0;
                if (prev == npieces - 1) p.counters[s] = 0;
            }
            csync();
            if (*last_flag) {
                // warp w folds pieces w, w + NW, ... into its running list, then the warps'
                // lists are merged
                for (int i = lane; i < Kp; i += 32) wbuf[i] = 0ull;
                uint64_t* scratch = wbuf + Kp;
                for (int32_t qq = warp; qq < npieces; qq += NW) {
                    const unsigned long long* src = reinterpret_cast<const unsigned long long*>(
                        p.slots + (int64_t)(c_first + qq + s) * K);
                    for (int i = lane; i < Kp; i += 32) scratch[i] = i < K ? __ldcg(src + i) : 0ull;
                    __syncwarp();
                    warp_merge_desc(wbuf, scratch, Kp, lane);
                }
                csync();
                merge_warps();
                finalize(s);
            }
        }
        csync();
        apos = pe;
    }
}

template <int D, int LPG>
int sel_prepare(uint32_t smem) {
    static int max_set = 0;
    if ((int)smem > max_set) {
        if (cudaFuncSetAttribute(page_select_kernel<D, LPG>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return -1;
        max_set = (int)smem;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, page_select_kernel<D, LPG>,
                                                      kSelWarps * 32, smem) != cudaSuccess)
        return 1;
    return n < 1 ? 1 : n;
}

template <int D, int LPG>
cudaError_t sel_go(int32_t G_req, int64_t units_bound, uint32_t smem, cudaStream_t stream,
                   SelParams& p, void* ws, size_t ws_bytes, bool& ws_ok) {
    const int occ = sel_prepare<D, LPG>(smem);
    if (occ < 0) return cudaErrorInvalidValue;
    const int32_t G = choose_splits(units_bound * 4, G_req, occ);
    const size_t counters = ((size_t)p.nseg * 4 + 255) & ~(size_t)255;
    ws_ok = !(ws == nullptr || ws_bytes < select_workspace_bytes(p.nseg, p.top_k, G) ||
              (reinterpret_cast<uintptr_t>(ws) & 255));
    if (!ws_ok) return cudaSuccess;
    p.counters = static_cast<int32_t*>(ws);
    p.slots = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(ws) + counters);
    return launch_pdl(page_select_kernel<D, LPG>, dim3(G), dim3(kSelWarps * 32), smem, stream, p);
}

template <int D>
cudaError_t sel_go_lpg(int lpg, int32_t G_req, int64_t units_bound, uint32_t smem,
                       cudaStream_t stream, SelParams& p, void* ws, size_t ws_bytes, bool& ok) {
    switch (lpg) {
        case 1: return sel_go<D, 1>(G_req, units_bound, smem, stream, p, ws, ws_bytes, ok);
        case 2: return sel_go<D, 2>(G_req, units_bound, smem, stream, p, ws, ws_bytes, ok);
        case 4: return sel_go<D, 4>(G_req, units_bound, smem, stream, p, ws, ws_bytes, ok);
        case 8: return sel_go<D, 8>(G_req, units_bound, smem, stream, p, ws, ws_bytes, ok);
        default: return sel_go<D, 16>(G_req, units_bound, smem, stream, p, ws, ws_bytes, ok);
    }
}

}  // namespace

size_t select_workspace_bytes(int32_t nseg, int32_t top_k, int32_t G) {
    const size_t counters = ((size_t)nseg * 4 + 255) & ~(size_t)255;
    return counters + (size_t)(G + nseg) * top_k * 8;
}

dattn_status_t launch_page_select(const dattn_kv_layout& Lay, const uint16_t* stats,
                                  const uint16_t* q, int32_t B, int32_t Hq,
                                  const int32_t* seq_lens, const int8_t* head_kind,
                                  int32_t top_k, int32_t* selected, int32_t* selected_phys,
                                  void* ws, size_t ws_bytes, int32_t num_splits,
                                  int32_t* dev_err, cudaStream_t stream, int64_t units_bound) {
    if (B == 0 || top_k == 0) return DATTN_OK;
    SelParams p{};
    p.num_pages = Lay.num_pages;
    p.Hkv = Lay.num_kv_heads;
    p.P = Lay.page_size;
    p.max_pages = Lay.max_pages_per_req;
    p.block_table = Lay.block_table;
    p.stats = stats;
    p.q = q;
    p.B = B;
    p.Hq = Hq;
    p.g = Hq / p.Hkv;
    p.seq_lens = seq_lens;
    p.head_kind = head_kind;
    p.top_k = top_k;
    p.selected = selected;
    p.selected_phys = selected_phys;
    p.nseg = B * p.Hkv;
    p.dev_err = dev_err;
    const int D = Lay.head_dim;
    const int lpg = p.P / 16;
    if (lpg & (lpg - 1)) return DATTN_ERR_UNSUPPORTED;  // P / 16 must be a power of two
    // one unit is 16 padded logical-page rows; up to three units in flight per warp, as
    // many as the shared memory of one CTA per SM holds
    const uint32_t stage_bytes = sel_stage_bytes(D, lpg);
    SelSmem L{};
    for (p.stages = 3; p.stages >= 1; --p.stages) {
        L = sel_smem_layout(B, p.Hkv, top_k, kSelWarps, stage_bytes, p.stages);
        if (L.total <= 227u * 1024u) break;
    }
    if (p.stages < 1) return DATTN_ERR_UNSUPPORTED;
    bool ws_ok = true;
    cudaError_t e;
    if (D == 64)
        e = sel_go_lpg<64>(lpg, num_splits, units_bound, L.total, stream, p, ws, ws_bytes, ws_ok);
    else
        e = sel_go_lpg<128>(lpg, num_splits, units_bound, L.total, stream, p, ws, ws_bytes,
                            ws_ok);
    if (!ws_ok) return DATTN_ERR_WORKSPACE;
    return e == cudaSuccess ? DATTN_OK : DATTN_ERR_CUDA;
}

}  // namespace dattn
