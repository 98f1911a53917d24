// Split-KV attention engine: MicroAttention partials over 16-token tiles and their
// log-sum-exp aggregation, for dattn_partial and for the dense and block-sparse dattn_decode.
//
// What it computes comes from "Infinite-LLM: Efficient LLM Service for Long Context with
// DistAttention and Distributed KVCache":
//   - "DistAttention 的等价数学变换": MicroAttention over a chunk of keys,
//       m_j = max s_i,  e_j = sum exp(s_i - m_j),  MA_j = sum exp(s_i - m_j) v_i;
//   - "结果聚合与通信开销降低": m_g = max m_j,  e_g = sum e_j exp(m_j - m_g),
//       out = sum MA_j exp(m_j - m_g) / e_g.
// The block-sparse token sets come from "LLM长序列服务优化：LServe的块稀疏注意力技术": §2.2.2
// (selected physical pages only) and §3.1.1 (sink tokens plus a local window for
// streaming heads, fused into the same kernel as the retrieval heads).
//
// GB300 design. The page tile of one (page, KV head) is contiguous in HBM. A producer warp
// streams 16-token K and V row groups into an 8-stage (8-bit pool: 12-stage) shared-memory
// ring with one 3-D TMA box each ({64, 16, d/64}: 128-byte swizzle, evict-first L2 policy,
// completion on mbarriers). Four consumer warps each own every fourth stage. A consumer
// runs the small QK^T tile with tokens as the M dimension and the GQA group as N (mma.sync
// m16n8k16, bf16 in, fp32 accumulate). It does an online softmax in base 2 with warp
// shuffles, transposes P with movmatrix, and accumulates O^T = V^T P^T with P split into
// two bf16 terms, so the weights keep 16 significant bits. The work of all (segment =
// request or chunk, KV head) pairs is laid end to end in 16-token tiles and cut into equal
// contiguous ranges, one per CTA. Each CTA therefore gets the same number of bytes,
// whatever the length mix. A segment that lies inside one CTA is finished there. A segment
// cut across CTAs leaves one partial triple per CTA in the workspace, and the CTA that
// arrives last (atomic counter) merges them. No CTA ever waits on another. The 8-bit pool
// (FP8 E4M3 codes with one fp32 scale per row) streams half the bytes through the same
// pipeline and runs on fp16 tensor cores (see Consumer).
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dattn {

namespace {

#define kNegInf (-__int_as_float(0x7f800000))

constexpr int kIssue = kConsumerWarps;  // tiles the producer issues side by side

struct Smem {
    uint8_t* base;
    AttnSmem L;
    __device__ uint32_t full_bar(int s) const { return smem_u32(base + L.bars) + 8u * s; }
    __device__ uint32_t empty_bar(int s) const {
        return smem_u32(base + L.bars) + 8u * (L.nstages + s);
    }
    __device__ int32_t* meta() const { return reinterpret_cast<int32_t*>(base + L.meta); }
    __device__ volatile int* abort_flag() const {
        return reinterpret_cast<volatile int*>(base + L.flags);
    }
    __device__ int* last_flag() const { return reinterpret_cast<int*>(base + L.flags + 4); }
    __device__ float* ws_m() const { return reinterpret_cast<float*>(base + L.ws_m); }
    __device__ float* ws_e() const { return reinterpret_cast<float*>(base + L.ws_e); }
    __device__ float* ws_o() const { return reinterpret_cast<float*>(base + L.ws_o); }
    __device__ int32_t* kind_before() const {
        return reinterpret_cast<int32_t*>(base + L.kind_before);
    }
    __device__ int32_t* kinds() const { return reinterpret_cast<int32_t*>(base + L.kinds); }
    __device__ int32_t* item_start() const {
        return reinterpret_cast<int32_t*>(base + L.item_start);
    }
    __device__ int32_t* item_len() const { return reinterpret_cast<int32_t*>(base + L.item_len); }
    // fused append: the position of request i's new token (its length before the append;
    // negative when nothing is appended)
    __device__ int32_t* item_pos() const { return reinterpret_cast<int32_t*>(base + L.item_pos); }
    // fused append, quantized pool: [warp][lane][3] codes and scale of the new row
    __device__ uint32_t* qrow() const { return reinterpret_cast<uint32_t*>(base + L.qrow); }
    // the CTA's plan constants: aligned, W, Gw, X0, X1
    __device__ int32_t* cplan() const { return reinterpret_cast<int32_t*>(base + L.flags + 8); }
    // head-aligned plan: kAplanScalars scalars, the retrieval heads, the streaming heads
    __device__ int32_t* aplan() const { return reinterpret_cast<int32_t*>(base + L.aplan); }
    __device__ int32_t* scan() const { return reinterpret_cast<int32_t*>(base + L.scan); }
    // the 8-bit pool's row scales of stage s: 16 K scales, then 16 V scales
    __device__ const float* scales(int s) const {
        return reinterpret_cast<const float*>(base + L.scales) + 32 * s;
    }
};


__device__ __forceinline__ int32_t ceil16(int32_t x) { return (x + 15) >> 4; }

// Tiles of a streaming head at length L: sink tiles, then the tiles of the local window.
__device__ __forceinline__ void stream_geometry(int32_t L, int32_t sinks, int32_t local,
                                                int32_t& s_end, int32_t& nsink, int32_t& l0,
                                                int32_t& nlocal) {
    s_end = min(sinks, L);
    nsink = ceil16(s_end);
    l0 = max(sinks, L - local);
    nlocal = (L > l0) ? ((L - 1) >> 4) - (l0 >> 4) + 1 : 0;
}

__device__ __forceinline__ int32_t head_tiles(int kind, int32_t L, const AttnParams& p) {
    if (kind == DATTN_HEAD_RETRIEVAL) return L > 0 ? p.top_k * (p.P >> 4) : 0;
    if (kind == DATTN_HEAD_STREAMING) {
        int32_t s_end, nsink, l0, nlocal;
        stream_geometry(L, p.sinks, p.local, s_end, nsink, l0, nlocal);
        return nsink + nlocal;
    }
    return ceil16(L);
}

// Every segment (one KV head of one request or chunk) is laid out in "cost units": its real
// 16-token tiles, then kSegCost units that stand for the fixed cost of a piece (fetching the
// query, merging the warps, handing over a partial). The balanced split cuts the cost space,
// so a CTA whose range crosses many small segments gets fewer tiles. The extra units are
// never loaded or scheduled: producer and consumers walk real tiles only.

// Head-aligned plan of a block-sparse launch in which every KV head is a retrieval or a
// streaming head. A retrieval segment then always holds R = top_k * P/16 tile slots and a
// streaming segment S = ceil(sinks/16) + ceil((local+15)/16) slots; the producer skips the
// slots the current length leaves empty. So the plan does not depend on the lengths and is
// made before the dependency wait. Each retrieval segment gets k CTAs of its own, which split
// its slots evenly: no CTA carries pieces of two retrieval segments, and every retrieval
// segment is merged from exactly k pieces. The other G - n_r k CTAs take the streaming
// segments, each whole. k follows the cost units of the balanced split (real tiles plus
// kSegCost per segment), rounded to the nearest integer, but leaves every streaming segment
// a CTA of its own when the grid allows: their pieces are short and bound by latency, and a
// CTA runs its pieces one after another.
enum AplanIdx : int { AP_ON = 0, AP_K, AP_GR, AP_GS, AP_NRET, AP_NSTR, AP_R, AP_S };

__device__ void make_aligned_plan(const AttnParams& p, const Smem& sm, int32_t G) {
    int32_t* a = sm.aplan();
    int32_t* ret = a + kAplanScalars;
    int32_t* str = ret + p.Hkv;
    int32_t nret = 0, nstr = 0, ndense = 0;
    for (int h = 0; h < p.Hkv; ++h) {
        const int k = sm.kinds()[h];
        if (k == DATTN_HEAD_RETRIEVAL) ret[nret++] = h;
        else if (k == DATTN_HEAD_STREAMING) str[nstr++] = h;
        else ++ndense;
    }
    const int32_t R = p.top_k * (p.P >> 4);
    const int32_t S = (p.sinks + 15) / 16 + (p.local > 0 ? (p.local + 30) / 16 : 0);
    const int64_t nr = (int64_t)p.B * nret, ns = (int64_t)p.B * nstr;
    int64_t k = 0;
    bool on = ndense == 0 && p.T == 1 && (nr > 0 || ns > 0) && (nret == 0 || R > 0) &&
              (nstr == 0 || S > 0);
    if (on && nr > 0) {
        const int64_t cr = R + kSegCost, cs = S + kSegCost;
        const int64_t W = nr * cr + ns * cs;
        k = (cr * G + W / 2) / W;
        k = min(max(k, (int64_t)1), (int64_t)R);
        // Streaming segments are short and bound by latency, so several in one CTA run one
        // after another: leave each its own CTA when the grid allows it, else at least one
        // CTA for all of them.
        if (ns > 0 && G - ns >= nr) k = min(k, ((int64_t)G - ns) / nr);
        k = min(k, (ns > 0 ? (int64_t)G - 1 : (int64_t)G) / nr);
        on = k >= 1;
    }
    a[AP_ON] = on ? 1 : 0;
    a[AP_K] = (int32_t)k;
    a[AP_GR] = (int32_t)(nr * k);
    a[AP_GS] = G - (int32_t)(nr * k);
    a[AP_NRET] = nret;
    a[AP_NSTR] = nstr;
    a[AP_R] = R;
    a[AP_S] = S;
}

// A piece: the real tiles [r0, r1) of segment s computed in this CTA. The segment's pieces
// lie in the consecutive CTAs cfirst .. clast (cfirst == clast: the segment is finished here).
struct Piece {
    int32_t s, r0, r1, cfirst, clast;
};

// Segment geometry derived from the per-item prefix sums (in cost units) in shared memory.
struct Plan {
    const AttnParams& p;
    const Smem& sm;
    __device__ Plan(const AttnParams& p_, const Smem& sm_) : p(p_), sm(sm_) {}

    __device__ static int32_t cost_of(int32_t real) { return real > 0 ? real + kSegCost : 0; }

    // Largest item i with item_start[i] <= t (t < W).
    __device__ int32_t item_of(int32_t t) const {
        const int32_t* st = sm.item_start();
        int32_t lo = 0, hi = p.nitems - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (st[mid] <= t) lo = mid; else hi = mid - 1;
        }
        return lo;
    }

    // Cost offset of head h within item i, its real tile count and its cost.
    __device__ void head_span(int32_t i, int32_t h, int32_t& off, int32_t& real,
                              int32_t& cost) const {
        if (p.mode == MODE_SPARSE) {
            const int32_t L = sm.item_len()[i];
            const int32_t n0 = head_tiles(DATTN_HEAD_DENSE, L, p);
            const int32_t n1 = head_tiles(DATTN_HEAD_RETRIEVAL, L, p);
            const int32_t n2 = head_tiles(DATTN_HEAD_STREAMING, L, p);
            const int32_t* kb = sm.kind_before() + 3 * h;
            off = kb[0] * cost_of(n0) + kb[1] * cost_of(n1) + kb[2] * cost_of(n2);
            const int k = sm.kinds()[h];
            real = k == DATTN_HEAD_RETRIEVAL ? n1 : (k == DATTN_HEAD_STREAMING ? n2 : n0);
        } else {
            // dense: item_len holds the length; partial: the real tiles per head
            real = p.mode == MODE_PARTIAL ? sm.item_len()[i] : ceil16(sm.item_len()[i]);
            off = h * cost_of(real);
        }
        cost = cost_of(real);
    }

    __device__ void seg_span(int32_t s, int32_t& start, int32_t& real, int32_t& cost) const {
        const int32_t i = s / p.Hkv, h = s - i * p.Hkv;
        int32_t off;
        head_span(i, h, off, real, cost);
        start = sm.item_start()[i] + off;
    }

    // Segment whose cost range contains position t (t < W).
    __device__ int32_t segment_at(int32_t t) const {
        const int32_t i = item_of(t);
        const int32_t o = t - sm.item_start()[i];
        int32_t lo = 0, hi = p.Hkv - 1;  // largest head whose offset is <= o
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            int32_t off, real, cost;
            head_span(i, mid, off, real, cost);
            if (off <= o) lo = mid; else hi = mid - 1;
        }
        return i * p.Hkv + lo;
    }

    // The next piece of the range [X0, X1) at or after segment s: the real tiles
    // [r0, r1) of segment s that fall in the range. Returns false when there is none.
    __device__ bool next_piece(int32_t& s, int32_t X0, int32_t X1, int32_t& cs, int32_t& real,
                               int32_t& r0, int32_t& r1) const {
        for (; s < p.nseg; ++s) {
            int32_t cost;
            seg_span(s, cs, real, cost);
            if (cs >= X1) return false;
            if (cost == 0) continue;
            r0 = max(X0 - cs, 0);
            r1 = min(X1 - cs, real);
            if (r0 < r1) return true;
        }
        return false;
    }
};

// The pieces of one CTA in order, under either plan. A cursor starts at 0; piece() returns
// the piece at the cursor, or false when there is none, and advance() moves past it.
// The CTA's constants of its plan sit in shared memory (sm.cplan(): aligned, W, Gw, X0, X1),
// so that they occupy no registers across the consumer loop.
struct PieceIter {
    const AttnParams& p;
    const Smem& sm;
    const Plan& plan;
    int32_t cta;
    __device__ PieceIter(const AttnParams& p_, const Smem& sm_, const Plan& pl, int32_t c)
        : p(p_), sm(sm_), plan(pl), cta(c) {}

    __device__ bool aligned() const { return sm.cplan()[0] != 0; }

    // Cursor: the segment to look from (balanced split) or the piece index (aligned plan).
    __device__ int32_t start() const {
        const int32_t* cp = sm.cplan();
        return cp[0] ? 0 : (cp[3] < cp[4] ? plan.segment_at(cp[3]) : p.nseg);
    }

    __device__ bool piece(int32_t& cur, Piece& pc) const {
        const int32_t* cp = sm.cplan();
        if (!cp[0]) {
            const int32_t W = cp[1], Gw = cp[2], X0 = cp[3], X1 = cp[4];
            int32_t cs, real, r0, r1;
            if (!plan.next_piece(cur, X0, X1, cs, real, r0, r1)) return false;
            pc.s = cur;
            pc.r0 = r0;
            pc.r1 = r1;
            pc.cfirst = split_owner(cs, W, Gw);
            pc.clast = split_owner(cs + real - 1, W, Gw);
            return true;
        }
        const int32_t* a = sm.aplan();
        const int32_t k = a[AP_K], Gr = a[AP_GR], Gs = a[AP_GS];
        if (cta < Gr) {
            if (cur != 0) return false;
            const int32_t r = cta / k, j = cta - r * k, R = a[AP_R], nret = a[AP_NRET];
            const int32_t b = r / nret;
            pc.s = b * p.Hkv + a[kAplanScalars + (r - b * nret)];
            pc.r0 = (int32_t)((int64_t)j * R / k);
            pc.r1 = (int32_t)((int64_t)(j + 1) * R / k);
            pc.cfirst = r * k;
            pc.clast = r * k + k - 1;
            return true;
        }
        const int32_t j = cta - Gr, nstr = a[AP_NSTR];
        const int64_t ns = (int64_t)p.B * nstr;
        if (j >= Gs || ns == 0) return false;
        const int64_t m = ns * j / Gs + cur;
        if (m >= ns * (j + 1) / Gs) return false;
        const int32_t b = (int32_t)(m / nstr);
        pc.s = b * p.Hkv + a[kAplanScalars + p.Hkv + (int32_t)(m - (int64_t)b * nstr)];
        pc.r0 = 0;
        pc.r1 = a[AP_S];
        pc.cfirst = pc.clast = cta;
        return true;
    }

    __device__ void advance(int32_t& cur) const { ++cur; }
};

// Resolved tile: TMA row coordinate, the valid token range [lo, hi) within its 16 rows and
// the causal cut of multi-query decode: row r is visible to query token t iff r <= cut + t.
// With the fused append, the tile that holds the new token carries its row: the consumer
// writes the new token's K and V into that row of the stage before using it.
// With the mixed pool, yc is the tile's row in its format's region (y, over all heads, still
// addresses the row scales) and kTileI4 marks a 4-bit tile.
struct TileRef {
    int32_t y;
    int32_t lohi;  // lo | hi << 8 | skip << 16 | patch << 17 | patch row << 18 | 4-bit << 22 |
                   // (cut + 16) << 24, cut clamped to [-16, 16]
    int32_t yc;
};
constexpr int32_t kTileSkip = 1 << 16;
constexpr int32_t kTilePatch = 1 << 17;
constexpr int32_t kTileI4 = 1 << 22;
__device__ __forceinline__ int32_t tile_lo(int32_t m) { return m & 0xff; }
__device__ __forceinline__ int32_t tile_hi(int32_t m) { return (m >> 8) & 0xff; }
__device__ __forceinline__ int32_t tile_cut(int32_t m) { return ((m >> 24) & 63) - 16; }
__device__ __forceinline__ int32_t tile_patch_row(int32_t m) { return (m >> 18) & 15; }

// Tile `local` of segment s. `aligned`: the head-aligned plan's fixed slot layout (streaming
// segments: ceil(sinks/16) sink slots, then the local-window slots; retrieval segments have
// slots even when the length is 0).
__device__ __forceinline__ TileRef resolve_tile(const AttnParams& p, const Smem& sm, int32_t s,
                                                int32_t local, bool aligned) {
    TileRef r{0, kTileSkip, 0};
    const int32_t item = s / p.Hkv, h = s - item * p.Hkv;
    int32_t b, L, t0, lo = 0, hi = 16, cut = 16;
    int32_t page = -2;  // -2: look the page up in the block table
    if (p.mode == MODE_PARTIAL) {
        b = __ldg(p.chunk_req + item);
        if (b < 0 || b >= p.B) return r;  // such a chunk has no tiles
        L = min(max(__ldg(p.seq_lens + b), 0), p.max_pages * p.P);
        const int32_t per_page = p.P >> 4;
        const int32_t pg = __ldg(p.chunk_pages + __ldg(p.chunk_indptr + item) + local / per_page);
        if (pg < 0 || pg >= p.max_pages) {
            set_err(p.dev_err, DATTN_DEVERR_CHUNK_OOB);
            return r;
        }
        t0 = pg * p.P + (local - (local / per_page) * per_page) * 16;
        if (t0 >= L) return r;
        hi = min(16, L - t0);
    } else {
        b = item;
        L = sm.item_len()[item];
        const int kind = p.mode == MODE_SPARSE ? sm.kinds()[h] : DATTN_HEAD_DENSE;
        if (kind == DATTN_HEAD_RETRIEVAL) {
            if (L == 0) return r;  // (aligned plan) nothing is attended
            const int32_t per_page = p.P >> 4;
            const int32_t si = local / per_page;
            const int64_t at = ((int64_t)b * p.Hkv + h) * p.top_k + si;
            const int32_t pg = __ldg(p.selected + at);
            if (p.selected_phys) page = __ldg(p.selected_phys + at);
            if (pg < 0) return r;
            if (pg >= (L + p.P - 1) / p.P) {
                set_err(p.dev_err, DATTN_DEVERR_SELECT_OOB);
                return r;
            }
            t0 = pg * p.P + (local - si * per_page) * 16;
            if (t0 >= L) return r;
            hi = min(16, L - t0);
        } else if (kind == DATTN_HEAD_STREAMING) {
            int32_t s_end, nsink, l0, nlocal;
            stream_geometry(L, p.sinks, p.local, s_end, nsink, l0, nlocal);
            int32_t j = local;  // the slot as a sink tile (j < nsink) or local tile j - nsink
            if (aligned) {
                const int32_t nsink_max = (p.sinks + 15) / 16;
                if (local < nsink_max) {
                    if (local >= nsink) return r;
                } else {
                    j = nsink + (local - nsink_max);
                    if (j - nsink >= nlocal) return r;
                }
            }
            if (j < nsink) {
                t0 = j * 16;
                hi = min(16, s_end - t0);
            } else {
                t0 = ((l0 >> 4) + (j - nsink)) * 16;
                lo = max(t0, l0) - t0;
                hi = min(t0 + 16, L) - t0;
            }
        } else {
            t0 = local * 16;
            hi = min(16, L - t0);
            // multi-query decode: query token t sees the tokens < L - T + t + 1
            if (p.T > 1) cut = min(16, max(-16, L - p.T - t0));
        }
    }
    const int32_t lp = t0 / p.P;
    if (page == -2) page = __ldg(p.block_table + (int64_t)b * p.max_pages + lp);
    if (page < 0) {
        set_err(p.dev_err, DATTN_DEVERR_UNMAPPED_PAGE);
        return r;
    }
    if (page >= p.num_pages) {
        set_err(p.dev_err, DATTN_DEVERR_PAGE_OOB);
        return r;
    }
    r.y = (page * p.Hkv + h) * p.P + (t0 - lp * p.P);
    r.lohi = lo | (hi << 8) | ((cut + 16) << 24);
    if (p.fmt == DATTN_KV_MIXED) {
        const bool i4 = head_is_i4(p.hf, h);
        const int32_t hc = i4 ? p.hf.h4 : p.Hkv - p.hf.h4;
        r.yc = (page * hc + head_class_index(p.hf, h, i4)) * p.P + (t0 - lp * p.P);
        if (i4) r.lohi |= kTileI4;
    }
    if (p.append) {  // the new token (the last one) lies in this tile
        const int32_t pos = sm.item_pos()[b];
        if (pos >= 0 && pos == L - 1 && pos >= t0 + lo && pos < t0 + hi)
            r.lohi |= kTilePatch | ((pos - t0) << 18);
    }
    return r;
}

// Writes the final result of column c of segment s: query token t = c / g of query head
// kvh*g + c % g. MA is unnormalised; m is in log2 units.
__device__ __forceinline__ void write_final(const AttnParams& p, int32_t s, int32_t c, int32_t d,
                                            int D, float m, float e, float ma) {
    const int32_t item = s / p.Hkv, kvh = s - item * p.Hkv;
    const int32_t t = c / p.g, j = c - t * p.g;
    const int64_t row = ((int64_t)item * p.T + t) * p.Hq + kvh * p.g + j;
    if (p.mode == MODE_PARTIAL) {
        p.out[row * D + d] = ma;
    } else {
        p.out[row * D + d] = e > 0.f ? ma / e : 0.f;
    }
    if (d == 0) {
        if (p.m_out) p.m_out[row] = m == kNegInf ? kNegInf : m * kLn2;
        if (p.e_out) p.e_out[row] = e;
    }
}

// The 8-bit pool (FP8 E4M3 codes with one fp32 scale per row) runs on fp16 tensor cores:
// every E4M3 value is an fp16 value, so a code converts exactly with one cvt per pair,
// straight from the ldmatrix fragment. The query is scaled by a power of two 2^a, chosen
// per piece so that its largest element lies in [2^14, 2^15), and rounded to fp16; this is
// exact for every element within 2^28 of the largest. The logit of row i is then
// (q' . code_i) * k_scale_i * scale * log2(e) * 2^-a. For PV the V scale of a row goes
// into its softmax weight: w_i = p_i * v_scale_i * 2^15 / r, where r is a power of two at
// least the largest V scale seen so far in the piece (raised, and the accumulator rescaled,
// when a tile brings a larger one). So 0 <= w_i <= 2^15 always fits fp16, and w_i is
// split into two fp16 terms (22 significant bits) as the bf16 path splits p_i. The
// accumulator is multiplied by r * 2^-15 when the piece is published.
// PK: 2 or 4 query columns over the 4-bit pool, whose PV weights take one product per m-tile
// (see tile_i4). (A mixed-pool instance would work the same way for its 4-bit heads.)
template <int D, int FMT, bool PK>
struct Consumer {
    static constexpr int KS = D / 16;  // k-steps of QK^T and m-tiles of PV
    static constexpr bool Q = FMT != DATTN_KV_BF16;  // a quantized pool with row scales
    static constexpr bool I4 = FMT == DATTN_KV_INT4;
    static constexpr bool MIX = FMT == DATTN_KV_MIXED;  // 8-bit or 4-bit per KV head
    static_assert(!I4 || Q, "the 4-bit pool is a quantized pool");
    static_assert(!MIX || Q, "the mixed pool is a quantized pool");
    static_assert(!PK || I4 || MIX, "packed columns are a 4-bit form");

    const AttnParams& p;
    const Smem& sm;
    const int warp, lane;
    uint32_t qf[KS][2];
    float o[KS][4];
    float m0, m1, e0, e1;
    float qsc;     // scale * log2(e) (quantized pools: times 2^-a; 4-bit: times 2^24) for the
                   // current piece's query
    int32_t rk;    // 8-bit pool: r = 2^rk bounds the V scales seen in this piece
    float rv, inv;  // 8-bit pool: r and 2^15 / r
    bool i4 = I4;   // the current piece's KV head is 4-bit (set per piece in a mixed pool)
    // 4-bit pool: 8 * 2^-24 * (sum of the query) of this lane's columns 2tig, 2tig + 1, and
    // the running sums of this lane's PV weights of those columns (see tile_i4)
    float qc[2] = {0.f, 0.f};
    float ws0 = 0.f, ws1 = 0.f;

    __device__ Consumer(const AttnParams& p_, const Smem& sm_, int w, int l)
        : p(p_), sm(sm_), warp(w), lane(l) {}

    // The query column whose queries column c carries: itself, except in a packed (PK) piece of
    // a 4-bit KV head (f4), whose columns repeat the queries of column c mod gq (tile_i4).
    __device__ __forceinline__ int dup_col(int c, bool f4) const {
        if constexpr (PK) {
            if (f4) return c & (p.gq - 1);
        }
        return c;
    }

    // Visibility of this lane's four logits (rows g8, g8 + 8; columns 2tig, 2tig + 1): the row
    // lies in [lo, hi) and, in a tile of multi-query decode that holds new tokens (cut < 15,
    // warp-uniform), row r is visible to column c's query token t = c / g iff r <= cut + t.
    __device__ __forceinline__ void visible(int lo, int hi, int cut, bool& a0, bool& a1,
                                            bool& a2, bool& a3) const {
        const int g8 = lane >> 2, tig = lane & 3;
        const bool v0 = g8 >= lo && g8 < hi, v1 = g8 + 8 >= lo && g8 + 8 < hi;
        a0 = a1 = v0;
        a2 = a3 = v1;
        if (cut < 15) {
            const bool f4 = MIX ? i4 : I4;
            const int tA = dup_col(2 * tig, f4) / p.g, tB = dup_col(2 * tig + 1, f4) / p.g;
            a0 = a0 && g8 <= cut + tA;
            a1 = a1 && g8 <= cut + tB;
            a2 = a2 && g8 + 8 <= cut + tA;
            a3 = a3 && g8 + 8 <= cut + tB;
        }
    }

    // Masks a quantized tile's logits (rows g8: s0, s1; g8 + 8: s2, s3) to -inf and its V
    // scales (vs0, vs1) to 0 where visible() hides them. Full tiles, the common case, skip it
    // (warp-uniform).
    __device__ __forceinline__ void mask_tile(int lo, int hi, int cut, float& s0, float& s1,
                                              float& s2, float& s3, float& vs0,
                                              float& vs1) const {
        if (lo > 0 || hi < 16 || cut < 15) {
            const int g8 = lane >> 2;
            bool a0, a1, a2, a3;
            visible(lo, hi, cut, a0, a1, a2, a3);
            s0 = a0 ? s0 : kNegInf;
            s1 = a1 ? s1 : kNegInf;
            s2 = a2 ? s2 : kNegInf;
            s3 = a3 ? s3 : kNegInf;
            vs0 = g8 >= lo && g8 < hi ? vs0 : 0.f;
            vs1 = g8 + 8 >= lo && g8 + 8 < hi ? vs1 : 0.f;
        }
    }

    // B fragments of the segment's query columns for segment s (column n = lane / 4 is query
    // token n / g of query head kvh*g + n % g), and the factor that turns a raw dot product
    // into a base-2 logit.
    __device__ void load_q(int32_t s, uint32_t (&dst)[KS][2], float& qs, float (&qcs)[2]) const {
        const int32_t item = s / p.Hkv, kvh = s - item * p.Hkv;
        int32_t b = item;
        if (p.mode == MODE_PARTIAL) b = __ldg(p.chunk_req + item);
        const bool f4 = MIX ? head_is_i4(p.hf, kvh) : I4;
        const int n = dup_col(lane >> 2, f4), tig = lane & 3;
        const bool ok = n < p.gq && b >= 0 && b < p.B;
        const int32_t t = ok ? n / p.g : 0, j = ok ? n - t * p.g : 0;
        const uint32_t* qv = reinterpret_cast<const uint32_t*>(
            p.q + (((int64_t)(ok ? b : 0) * p.T + t) * p.Hq + kvh * p.g + j) * D);
        if constexpr (!Q) {
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                dst[ks][0] = ok ? __ldg(qv + ks * 8 + tig) : 0u;
                dst[ks][1] = ok ? __ldg(qv + ks * 8 + 4 + tig) : 0u;
            }
            qs = p.sl2;
            qcs[0] = qcs[1] = 0.f;
        } else {
            // The channels come in the order the quantized K fragment brings them.
            // 8-bit: k-step ks covers channels 16ks..16ks+15, b0 = 16ks + 4tig + {0, 1},
            // b1 = 16ks + 4tig + {2, 3}.
            // 4-bit: k-step ks takes channels c0 + {0..7} of the 32-channel chunk ks / 2,
            // c0 = 32 (ks / 2) + 8tig, in nibble pairs: sub-step ks % 2 = 0 has b0 = c0 + {0, 4}
            // and b1 = c0 + {1, 5}, sub-step 1 has b0 = c0 + {2, 6} and b1 = c0 + {3, 7}.
            float mx = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                if (f4) {
                    const uint4 w = ok ? __ldg(reinterpret_cast<const uint4*>(qv + (ks >> 1) * 16 +
                                                                             4 * tig))
                                       : make_uint4(0u, 0u, 0u, 0u);
                    const uint32_t e = (ks & 1) ? w.y : w.x, o4 = (ks & 1) ? w.w : w.z;
                    dst[ks][0] = __byte_perm(e, o4, 0x5410);
                    dst[ks][1] = __byte_perm(e, o4, 0x7632);
                } else {
                    dst[ks][0] = ok ? __ldg(qv + ks * 8 + 2 * tig) : 0u;
                    dst[ks][1] = ok ? __ldg(qv + ks * 8 + 2 * tig + 1) : 0u;
                }
                mx = fmaxf(mx, fmaxf(fmaxf(fabsf(bf16_lo(dst[ks][0])), fabsf(bf16_hi(dst[ks][0]))),
                                     fmaxf(fabsf(bf16_lo(dst[ks][1])), fabsf(bf16_hi(dst[ks][1])))));
            }
#pragma unroll
            for (int off = 1; off < 32; off <<= 1)
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            int32_t a = 0;  // 2^a * max|q| in [2^14, 2^15)
            if (mx > 0.f) a = min(127, max(-113, 14 - (((__float_as_int(mx) >> 23) & 0xff) - 127)));
            const float up = __int_as_float((127 + a) << 23);
            const float down = a < 127 ? __int_as_float((127 - a) << 23) : 5.877471754e-39f;
            // 4-bit: b1 meets the odd nibbles, which convert to 16 n * 2^-24 (i4pair_raw), so
            // its query values are divided by 16 (exact for elements within 2^24 of the
            // largest); qsum adds the values the products use, each odd one times 16
            const float up1 = f4 ? up * 0.0625f : up;
            float qsum = 0.f;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                dst[ks][0] = pack_f16(bf16_lo(dst[ks][0]) * up, bf16_hi(dst[ks][0]) * up);
                dst[ks][1] = pack_f16(bf16_lo(dst[ks][1]) * up1, bf16_hi(dst[ks][1]) * up1);
                if (f4)
                    qsum += (f16_lo(dst[ks][0]) + f16_hi(dst[ks][0])) +
                            16.f * (f16_lo(dst[ks][1]) + f16_hi(dst[ks][1]));
            }
            // 4-bit: times 2^24, the scale of the subnormal codes (exact)
            qs = f4 ? (p.sl2 * down) * 16777216.f : p.sl2 * down;
            qcs[0] = qcs[1] = 0.f;
            if (f4) {
                // the sum of column g8 over its four lanes, then columns 2tig, 2tig + 1
                qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
                qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
                qcs[0] = __shfl_sync(0xffffffffu, qsum, 8 * tig) * 4.76837158203125e-07f;
                qcs[1] = __shfl_sync(0xffffffffu, qsum, 8 * tig + 4) * 4.76837158203125e-07f;
            }
        }
    }

    // Fused append: this lane's 16-byte chunk of segment s's new K / V row (lanes 0 .. D/8 - 1
    // hold the K chunks, lanes D/8 .. D/4 - 1 the V chunks).
    __device__ uint4 load_new_row(int32_t s) const {
        constexpr int VPR = D / 8;
        const int32_t item = s / p.Hkv, kvh = s - item * p.Hkv;
        if (lane >= 2 * VPR || sm.item_pos()[item] < 0) return make_uint4(0u, 0u, 0u, 0u);
        const uint16_t* src = (lane < VPR ? p.k_new : p.v_new) +
                              ((int64_t)item * p.Hkv + kvh) * D + (lane % VPR) * 8;
        return __ldg(reinterpret_cast<const uint4*>(src));
    }

    // Fused append, quantized pool: this lane's codes of segment s's new K or V row (8-bit: 8
    // bytes; 4-bit: 4 bytes) and the row's scale, quantized exactly as the write half
    // quantizes them (the row maxima reduced over the lanes of each row; lanes as in
    // load_new_row). Computed when a piece starts and kept in the warp's shared memory (not in
    // registers, which the tile loop needs), for store_row_q.
    __device__ void quant_new_row(int32_t s, bool f4) const {
        constexpr int VPR = D / 8;
        const uint4 v = load_new_row(s);  // zero for lanes past the two rows
        float m = absmax8(v);
#pragma unroll
        for (int off = 1; off < VPR; off <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
        uint32_t* r = sm.qrow() + (warp * 32 + lane) * 3;
        float scale;
        if (f4) {
            r[0] = quant4_chunk(v, m, scale);
            r[1] = 0u;
        } else {
            const uint2 c = quant8_chunk(v, m, scale);
            r[0] = c.x;
            r[1] = c.y;
        }
        r[2] = __float_as_uint(scale);
    }

    // Writes this lane's codes (from quant_new_row) into row `row` of the quantized stage `st`
    // (8-bit, or 4-bit when f4), in the layout the TMA boxes leave there, and the rows' scales
    // into the stage's scales `sc`.
    __device__ void store_row_q(uint32_t st, float* sc, int row, bool f4) const {
        constexpr int VPR = D / 8;
        if (lane < 2 * VPR) {
            const uint32_t* r = sm.qrow() + (warp * 32 + lane) * 3;
            const bool isv = lane >= VPR;
            const int c8 = lane % VPR;
            if (f4)
                st_shared_u32(st + (isv ? 8u * D : 0u) + swz_rows<D / 2>((uint32_t)row, c8 >> 2) +
                                  (uint32_t)(c8 & 3) * 4u,
                              r[0]);
            else
                st_shared_v2(st + (isv ? 16u * D : 0u) + swz_rows<D>((uint32_t)row, c8 >> 1) +
                                 (uint32_t)(c8 & 1) * 8u,
                             r[0], r[1]);
            if (c8 == 0) sc[(isv ? 16 : 0) + row] = __uint_as_float(r[2]);
        }
        __syncwarp();
    }

    // Writes the new token's K and V (this lane's chunk v from load_new_row) into row `row` of
    // the bf16 stage `st`, in the layout the TMA boxes leave there.
    __device__ void patch_row(uint32_t st, int row, const uint4& v) const {
        constexpr int VPR = D / 8;
        if (lane < 2 * VPR) {
            const uint32_t c = (uint32_t)(lane % VPR);
            const uint32_t half0 = lane < VPR ? 0u : (uint32_t)(D / 64) * 2048u;
            st_shared_v4(st + half0 + (c >> 3) * 2048u + swz128((uint32_t)row, c & 7u), v);
        }
        __syncwarp();
    }

    __device__ void reset() {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        m0 = m1 = kNegInf;
        e0 = e1 = 0.f;
        ws0 = ws1 = 0.f;
        rk = -112;
        rv = __int_as_float((127 - 112) << 23);
        inv = __int_as_float((142 + 112) << 23);
    }

    // Online softmax (base 2) over one tile's logits: rows g8 (s0, s1) and g8 + 8 (s2, s3),
    // heads 2tig and 2tig + 1. Returns the weights relative to the new running max.
    __device__ __forceinline__ void softmax(float s0, float s1, float s2, float s3, float& p0,
                                            float& p1, float& p2, float& p3) {
        // the columns' maxima over the warp are needed only when some lane's logits exceed
        // the running maxima (rarely, once a piece is under way); otherwise they stay
        float c0 = fmaxf(s0, s2), c1 = fmaxf(s1, s3);
        float mn0 = m0, mn1 = m1;
        const bool raise = __any_sync(0xffffffffu, c0 > m0 || c1 > m1);
        if (raise) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                c0 = fmaxf(c0, __shfl_xor_sync(0xffffffffu, c0, off));
                c1 = fmaxf(c1, __shfl_xor_sync(0xffffffffu, c1, off));
            }
            mn0 = fmaxf(m0, c0);
            mn1 = fmaxf(m1, c1);
        }
        const float mu0 = mn0 == kNegInf ? 0.f : mn0, mu1 = mn1 == kNegInf ? 0.f : mn1;
        p0 = ex2_approx(s0 - mu0);
        p1 = ex2_approx(s1 - mu1);
        p2 = ex2_approx(s2 - mu0);
        p3 = ex2_approx(s3 - mu1);
        if (raise) {
            const float al0 = ex2_approx(m0 - mu0), al1 = ex2_approx(m1 - mu1);
            e0 *= al0;
            e1 *= al1;
            float alo = al1;  // the factor of O's column 1
            if constexpr (I4 || MIX) {
                ws0 *= al0;
                ws1 *= al1;
            }
            if constexpr (Q) {
                if (p.gq == 1) alo = al0;  // column 1 holds column 0's lo terms (g1_weights)
            }
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                o[mt][0] *= al0; o[mt][1] *= alo; o[mt][2] *= al0; o[mt][3] *= alo;
            }
        }
        m0 = mn0;
        m1 = mn1;
        e0 += p0 + p2;
        e1 += p1 + p3;
    }

    // One 16-token tile in stage buffer `st`; rows outside [lo, hi) are masked, and row r is
    // masked for query token t when r > cut + t.
    __device__ void tile(uint32_t st, int lo, int hi, int cut) {
        const uint32_t kbase = st, vbase = st + (uint32_t)(D / 64) * 2048u;
        // ---- S^T = K Q^T (tokens x heads) -------------------------------------------
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const uint32_t row = (lane & 7) + ((lane >> 3) & 1) * 8;
            const uint32_t csel = lane >> 4;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const uint32_t chunk = 2u * ks + csel;
                const uint32_t addr = kbase + (chunk >> 3) * 2048u + swz128(row, chunk & 7u);
                uint32_t a0, a1, a2, a3;
                ldsm_x4(addr, a0, a1, a2, a3);
                if (ks & 1) mma_bf16(sb, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
                else        mma_bf16(sa, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
            }
        }
        bool a0, a1, a2, a3;
        visible(lo, hi, cut, a0, a1, a2, a3);
        const float s0 = a0 ? (sa[0] + sb[0]) * qsc : kNegInf;
        const float s1 = a1 ? (sa[1] + sb[1]) * qsc : kNegInf;
        const float s2 = a2 ? (sa[2] + sb[2]) * qsc : kNegInf;
        const float s3 = a3 ? (sa[3] + sb[3]) * qsc : kNegInf;
        float p0, p1, p2, p3;
        softmax(s0, s1, s2, s3, p0, p1, p2, p3);
        // ---- P^T as the B operand: two bf16 terms, transposed with movmatrix ---------
        const uint32_t h01 = pack_bf16(p0, p1), h23 = pack_bf16(p2, p3);
        const uint32_t l01 = pack_bf16(p0 - bf16_lo(h01), p1 - bf16_hi(h01));
        const uint32_t l23 = pack_bf16(p2 - bf16_lo(h23), p3 - bf16_hi(h23));
        const uint32_t bh0 = movmatrix_trans(h01), bh1 = movmatrix_trans(h23);
        const uint32_t bl0 = movmatrix_trans(l01), bl1 = movmatrix_trans(l23);
        // ---- masked rows of V are zeroed so that 0 * (stale data) cannot give NaN -----
        if (lo > 0 || hi < 16) {
            const int nz = 16 - (hi - lo);
            for (int idx = lane; idx < nz * 8 * (D / 64); idx += 32) {
                const int rr = idx / (8 * (D / 64));
                const int rem = idx - rr * 8 * (D / 64);
                const int half = rem >> 3, ch = rem & 7;
                const int row = rr < lo ? rr : hi + (rr - lo);
                uint8_t* ptr = sm.base + (vbase - smem_u32(sm.base)) + half * 2048 +
                               swz128(row, ch);
                *reinterpret_cast<uint4*>(ptr) = make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
        }
        // ---- O^T += V^T P^T ----------------------------------------------------------
        {
            const uint32_t j = lane >> 3;
            const uint32_t row = (lane & 7) + (j >> 1) * 8;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                const uint32_t chunk = 2u * mt + (j & 1);
                const uint32_t addr = vbase + (chunk >> 3) * 2048u + swz128(row, chunk & 7u);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_trans(addr, a0, a1, a2, a3);
                mma_bf16(o[mt], a0, a1, a2, a3, bh0, bh1);
                mma_bf16(o[mt], a0, a1, a2, a3, bl0, bl1);
            }
        }
    }

    // One 16-token tile of the 8-bit pool in stage buffer `st` (K codes, then V codes) with
    // its row scales `sc`; rows are masked as in tile().
    __device__ void tile_f8(uint32_t st, const float* sc, int lo, int hi, int cut) {
        const uint32_t kbase = st, vbase = st + 16u * D;
        const int g8 = lane >> 2, tig = lane & 3;
        // ldmatrix lane addresses: matrices (rows 0-7 | 8-15) x (chunk 2c | 2c + 1)
        const uint32_t row = (lane & 7) + ((lane >> 3) & 1) * 8;
        const uint32_t csel = lane >> 4;
        // ---- S^T = K Q^T: a thread's 4 codes are 4 adjacent channels of one token ------
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t r0, r1, r2, r3, a0, a1, a2, a3;
            ldsm_x4(kbase + swz_rows<D>(row, 2u * c + csel), r0, r1, r2, r3);
            e4m3x4_to_f16(r0, a0, a2);
            e4m3x4_to_f16(r1, a1, a3);
            mma_f16(sa, a0, a1, a2, a3, qf[2 * c][0], qf[2 * c][1]);
            e4m3x4_to_f16(r2, a0, a2);
            e4m3x4_to_f16(r3, a1, a3);
            mma_f16(sb, a0, a1, a2, a3, qf[2 * c + 1][0], qf[2 * c + 1][1]);
        }
        const float kc0 = sc[g8] * qsc, kc1 = sc[g8 + 8] * qsc;
        float s0 = (sa[0] + sb[0]) * kc0, s1 = (sa[1] + sb[1]) * kc0;
        float s2 = (sa[2] + sb[2]) * kc1, s3 = (sa[3] + sb[3]) * kc1;
        float vs0 = sc[16 + g8], vs1 = sc[24 + g8];
        mask_tile(lo, hi, cut, s0, s1, s2, s3, vs0, vs1);
        float p0, p1, p2, p3;
        softmax(s0, s1, s2, s3, p0, p1, p2, p3);
        // ---- V scales: raise r to a power of two >= every V scale of the tile ---------
        raise_r(fmaxf(vs0, vs1));
        const float vn0 = vs0 * inv, vn1 = vs1 * inv;  // in [0, 2^15], exact
        const float w0 = p0 * vn0, w1 = p1 * vn0, w2 = p2 * vn1, w3 = p3 * vn1;
        // ---- W^T as the B operand: two fp16 terms, transposed with movmatrix ----------
        // (one query column: both terms in one operand, one product per m-tile)
        const bool g1 = p.gq == 1;
        uint32_t bh0, bh1, bl0 = 0u, bl1 = 0u;
        if (g1) {
            g1_weights(w0, w2, bh0, bh1);
        } else {
            const uint32_t h01 = pack_f16(w0, w1), h23 = pack_f16(w2, w3);
            const uint32_t l01 = pack_f16(w0 - f16_lo(h01), w1 - f16_hi(h01));
            const uint32_t l23 = pack_f16(w2 - f16_lo(h23), w3 - f16_hi(h23));
            bh0 = movmatrix_trans(h01);
            bh1 = movmatrix_trans(h23);
            bl0 = movmatrix_trans(l01);
            bl1 = movmatrix_trans(l23);
        }
        // ---- O^T += V^T W^T ------------------------------------------------------------
        // After the transposing ldmatrix a thread holds tokens 2tig, 2tig + 1 (or 8 + ...)
        // of channels 2g8, 2g8 + 1 of a 16-channel chunk; codes of masked tokens are zeroed
        // so that a stale NaN code cannot meet a zero weight. Row g8 of m-tile mt is
        // channel 16mt + 2g8 and row g8 + 8 is channel 16mt + 2g8 + 1.
        uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
        if (lo > 0 || hi < 16) {
            const int t0 = 2 * tig, t1 = 2 * tig + 1;
            mlo = (t0 >= lo && t0 < hi ? 0x0000ffffu : 0u) | (t1 >= lo && t1 < hi ? 0xffff0000u : 0u);
            mhi = (t0 + 8 >= lo && t0 + 8 < hi ? 0x0000ffffu : 0u) |
                  (t1 + 8 >= lo && t1 + 8 < hi ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t r0, r1, r2, r3, a0, a1, a2, a3;
            ldsm_x4_trans(vbase + swz_rows<D>(row, 2u * c + csel), r0, r1, r2, r3);
            // [t0 cA, t0 cB, t1 cA, t1 cB] -> [t0 cA, t1 cA, t0 cB, t1 cB]
            r0 = __byte_perm(r0 & mlo, 0u, 0x3120);
            r1 = __byte_perm(r1 & mhi, 0u, 0x3120);
            r2 = __byte_perm(r2 & mlo, 0u, 0x3120);
            r3 = __byte_perm(r3 & mhi, 0u, 0x3120);
            e4m3x4_to_f16(r0, a0, a1);
            e4m3x4_to_f16(r1, a2, a3);
            mma_f16(o[2 * c], a0, a1, a2, a3, bh0, bh1);
            if (!g1) mma_f16(o[2 * c], a0, a1, a2, a3, bl0, bl1);
            e4m3x4_to_f16(r2, a0, a1);
            e4m3x4_to_f16(r3, a2, a3);
            mma_f16(o[2 * c + 1], a0, a1, a2, a3, bh0, bh1);
            if (!g1) mma_f16(o[2 * c + 1], a0, a1, a2, a3, bl0, bl1);
        }
    }

    // ---- 4-bit pool ------------------------------------------------------------------
    // A tile in a stage buffer is K codes then V codes, rows of d/2 bytes (two codes per
    // byte), with its row scales in `sc`; the scales enter exactly as in tile_f8, and every
    // code converts exactly to fp16.

    // S^T = K Q^T of one tile into two accumulator chains: a thread's ldmatrix register holds
    // 8 adjacent channels of one token, and nibble pairs (k, k + 4) form the fragments in the
    // order load_q takes the query.
    __device__ __forceinline__ void qk_i4(uint32_t kbase, float (&sa)[4], float (&sb)[4]) const {
        constexpr uint32_t RB = D / 2;
        // ldmatrix lane addresses: matrices (rows 0-7 | 8-15) x (chunk 2c | 2c + 1)
        const uint32_t row = (lane & 7) + ((lane >> 3) & 1) * 8;
        const uint32_t csel = lane >> 4;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
            uint32_t r0, r1, r2, r3;  // chunk 2c: tokens g8, g8 + 8; chunk 2c + 1: the same
            ldsm_x4(kbase + swz_rows<RB>(row, 2u * c + csel), r0, r1, r2, r3);
            mma_f16(sa, i4pair_raw<0>(r0), i4pair_raw<0>(r1), i4pair_raw<1>(r0),
                    i4pair_raw<1>(r1), qf[4 * c][0], qf[4 * c][1]);
            mma_f16(sb, i4pair_raw<2>(r0), i4pair_raw<2>(r1), i4pair_raw<3>(r0),
                    i4pair_raw<3>(r1), qf[4 * c + 1][0], qf[4 * c + 1][1]);
            mma_f16(sa, i4pair_raw<0>(r2), i4pair_raw<0>(r3), i4pair_raw<1>(r2),
                    i4pair_raw<1>(r3), qf[4 * c + 2][0], qf[4 * c + 2][1]);
            mma_f16(sb, i4pair_raw<2>(r2), i4pair_raw<2>(r3), i4pair_raw<3>(r2),
                    i4pair_raw<3>(r3), qf[4 * c + 3][0], qf[4 * c + 3][1]);
        }
    }

    // Raises r to a power of two >= every lane's vl (the largest V scale of its rows), rescaling
    // O (and the 4-bit weight sums). The maximum over the warp is taken only when some lane's
    // exceeds r.
    __device__ __forceinline__ void raise_r(float vl) {
        if (__any_sync(0xffffffffu, vl > rv)) {
            const float vt = warp_vmax(vl);  // > r >= 2^-112: a normal number
            const int32_t bits = __float_as_int(vt);
            const int32_t k = min(127, ((bits >> 23) & 0xff) - 127 + ((bits & 0x7fffff) != 0));
            const int32_t dk = rk - k;
            const float f = dk >= -126 ? __int_as_float((127 + dk) << 23) : 0.f;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                o[mt][0] *= f; o[mt][1] *= f; o[mt][2] *= f; o[mt][3] *= f;
            }
            ws0 *= f;
            ws1 *= f;
            rk = k;
            rv = __int_as_float((127 + k) << 23);
            inv = __int_as_float((142 - k) << 23);
        }
    }

    // O^T += V^T W^T for one tile with this lane's weights (rows g8: w0, w1; g8 + 8: w2, w3).
    // After the transposing ldmatrix a thread holds tokens 2tig, 2tig + 1 (r0, r2) or
    // 8 + 2tig, 9 + 2tig (r1, r3) of channels 4g8 .. 4g8 + 3 of a 32-channel chunk, and nibble
    // k of both halves is channel 4g8 + k of the two tokens: exactly an A fragment. M-tile mt
    // takes channels 32 (mt / 2) + 4g8 + 2 (mt % 2) + {0, 1} as its rows g8 and g8 + 8. Every
    // code is a finite value, so a masked row (weight 0) needs no zeroing.
    // The weights enter as two fp16 terms, hi and lo. With 8 query columns (kPvTwo) each m-tile
    // takes two products, one per term. One query column (kPvOne, as in MHA decode): the hi
    // and lo terms of column 0's weights (rows g8: w0, g8 + 8: w2) as columns 0 and 1 of one B
    // operand (g1_weights), so that each m-tile takes one product; column 1 of the accumulator
    // is then the lo part of column 0, rescaled with it and added to it when the piece is
    // published. 2 or 4 query columns (kPvPacked, a PK consumer): every column carries the
    // queries of column c mod gq (dup_col), so the lanes of columns c and c + gq hold the same
    // logits, running maxima and weights; columns [0, gq) take the hi terms and [gq, 2gq) the
    // lo terms, again one product per m-tile, and the accumulator's columns [gq, 2gq), rescaled
    // exactly as columns [0, gq), are added to them at publish.
    __device__ __forceinline__ void g1_weights(float w0, float w2, uint32_t& b0,
                                               uint32_t& b1) const {
        const float h0 = __half2float(__float2half_rn(w0)), h2 = __half2float(__float2half_rn(w2));
        const bool c0 = (lane & 3) == 0;  // the lanes of column 0
        b0 = movmatrix_trans(c0 ? pack_f16(h0, w0 - h0) : 0u);
        b1 = movmatrix_trans(c0 ? pack_f16(h2, w2 - h2) : 0u);
    }

    static constexpr int kPvTwo = 0, kPvOne = 1, kPvPacked = 2;
    template <int M>
    __device__ __forceinline__ void pv_i4(uint32_t vbase, float w0, float w1, float w2,
                                          float w3) {
        constexpr uint32_t RB = D / 2;
        constexpr bool G1 = M != kPvTwo;  // one product per m-tile
        const uint32_t row = (lane & 7) + ((lane >> 3) & 1) * 8;
        const uint32_t csel = lane >> 4;
        // W^T as the B operand: two fp16 terms, transposed with movmatrix
        uint32_t bh0, bh1, bl0 = 0u, bl1 = 0u;
        if constexpr (M == kPvOne) {
            g1_weights(w0, w2, bh0, bh1);
        } else if constexpr (M == kPvPacked) {
            const uint32_t h01 = pack_f16(w0, w1), h23 = pack_f16(w2, w3);
            const uint32_t l01 = pack_f16(w0 - f16_lo(h01), w1 - f16_hi(h01));
            const uint32_t l23 = pack_f16(w2 - f16_lo(h23), w3 - f16_hi(h23));
            const int c0 = 2 * (lane & 3);  // this lane's columns c0, c0 + 1 (gq = 2 or 4)
            const bool hi = c0 < p.gq, lo = !hi && c0 < 2 * p.gq;
            bh0 = movmatrix_trans(hi ? h01 : lo ? l01 : 0u);
            bh1 = movmatrix_trans(hi ? h23 : lo ? l23 : 0u);
        } else {
            const uint32_t h01 = pack_f16(w0, w1), h23 = pack_f16(w2, w3);
            const uint32_t l01 = pack_f16(w0 - f16_lo(h01), w1 - f16_hi(h01));
            const uint32_t l23 = pack_f16(w2 - f16_lo(h23), w3 - f16_hi(h23));
            bh0 = movmatrix_trans(h01);
            bh1 = movmatrix_trans(h23);
            bl0 = movmatrix_trans(l01);
            bl1 = movmatrix_trans(l23);
        }
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4_trans(vbase + swz_rows<RB>(row, 2u * c + csel), r0, r1, r2, r3);
            {
                const uint32_t x0 = i4pair_raw<0>(r0), x1 = i4pair_raw<1>(r0);
                const uint32_t x2 = i4pair_raw<0>(r1), x3 = i4pair_raw<1>(r1);
                mma_f16(o[4 * c], x0, x1, x2, x3, bh0, bh1);
                if constexpr (!G1) mma_f16(o[4 * c], x0, x1, x2, x3, bl0, bl1);
            }
            {
                const uint32_t x0 = i4pair_raw<2>(r0), x1 = i4pair_raw<3>(r0);
                const uint32_t x2 = i4pair_raw<2>(r1), x3 = i4pair_raw<3>(r1);
                mma_f16(o[4 * c + 1], x0, x1, x2, x3, bh0, bh1);
                if constexpr (!G1) mma_f16(o[4 * c + 1], x0, x1, x2, x3, bl0, bl1);
            }
            {
                const uint32_t x0 = i4pair_raw<0>(r2), x1 = i4pair_raw<1>(r2);
                const uint32_t x2 = i4pair_raw<0>(r3), x3 = i4pair_raw<1>(r3);
                mma_f16(o[4 * c + 2], x0, x1, x2, x3, bh0, bh1);
                if constexpr (!G1) mma_f16(o[4 * c + 2], x0, x1, x2, x3, bl0, bl1);
            }
            {
                const uint32_t x0 = i4pair_raw<2>(r2), x1 = i4pair_raw<3>(r2);
                const uint32_t x2 = i4pair_raw<2>(r3), x3 = i4pair_raw<3>(r3);
                mma_f16(o[4 * c + 3], x0, x1, x2, x3, bh0, bh1);
                if constexpr (!G1) mma_f16(o[4 * c + 3], x0, x1, x2, x3, bl0, bl1);
            }
        }
    }

    // Largest V scale of this lane's visible rows, reduced over the warp's row groups.
    __device__ __forceinline__ float warp_vmax(float v) const {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
        return v;
    }

    // One tile of the 4-bit pool; rows are masked as in tile(). The codes enter the products
    // as n * 2^-24 (n = code + 8; odd nibbles 16 n * 2^-24 against a query divided by 16), so
    // the raw products are 2^-24 (q' . n): the logit subtracts 8 * 2^-24 * (sum of q') (qc)
    // and scales by 2^24 (in qsc); the PV accumulator's offset, 8 * 2^-24 * (sum of the weights), is
    // taken out when the piece is published (ws0, ws1 keep those sums). Both corrections are
    // of the size of the values they correct, so nothing cancels catastrophically.
    __device__ void tile_i4(uint32_t st, const float* sc, int lo, int hi, int cut) {
        const int g8 = lane >> 2;
        // the offset correction -qc enters as the products' initial accumulator
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        qk_i4(st, sa, sb);
        const float kc0 = sc[g8] * qsc, kc1 = sc[g8 + 8] * qsc;  // qsc carries the codes' 2^24
        float s0 = ((sa[0] + sb[0]) - qc[0]) * kc0, s1 = ((sa[1] + sb[1]) - qc[1]) * kc0;
        float s2 = ((sa[2] + sb[2]) - qc[0]) * kc1, s3 = ((sa[3] + sb[3]) - qc[1]) * kc1;
        float vs0 = sc[16 + g8], vs1 = sc[24 + g8];
        mask_tile(lo, hi, cut, s0, s1, s2, s3, vs0, vs1);
        float p0, p1, p2, p3;
        softmax(s0, s1, s2, s3, p0, p1, p2, p3);
        raise_r(fmaxf(vs0, vs1));
        const float vn0 = vs0 * inv, vn1 = vs1 * inv;  // in [0, 2^15], exact
        const float w0 = p0 * vn0, w1 = p1 * vn0, w2 = p2 * vn1, w3 = p3 * vn1;
        ws0 += w0 + w2;
        ws1 += w1 + w3;
        if constexpr (PK)  pv_i4<kPvPacked>(st + 8u * D, w0, w1, w2, w3);
        else if (p.gq == 1) pv_i4<kPvOne>(st + 8u * D, w0, w1, w2, w3);
        else               pv_i4<kPvTwo>(st + 8u * D, w0, w1, w2, w3);
    }

    // Publishes this warp's state for the CTA-level merge of the piece.
    __device__ void publish() {
        float t0 = e0, t1 = e1;
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            t0 += __shfl_xor_sync(0xffffffffu, t0, off);
            t1 += __shfl_xor_sync(0xffffffffu, t1, off);
        }
        const int g8 = lane >> 2, tig = lane & 3;
        const int hA = 2 * tig, hB = 2 * tig + 1;
        float* wm = sm.ws_m() + warp * kMaxGroup;
        float* we = sm.ws_e() + warp * kMaxGroup;
        float* wo = sm.ws_o() + warp * p.gq * D;
        if (g8 == 0) {
            if (hA < p.gq) { wm[hA] = m0; we[hA] = t0; }
            if (hB < p.gq) { wm[hB] = m1; we[hB] = t1; }
        }
        if constexpr (!Q) {
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                const int dd = mt * 16 + g8;
                if (hA < p.gq) { wo[hA * D + dd] = o[mt][0]; wo[hA * D + dd + 8] = o[mt][2]; }
                if (hB < p.gq) { wo[hB * D + dd] = o[mt][1]; wo[hB * D + dd + 8] = o[mt][3]; }
            }
        } else {
            const float rs = rv * 3.0517578125e-05f;  // r * 2^-15, exact
            const bool f4 = MIX ? i4 : I4;
            // 4-bit: row g8 of an m-tile (an even nibble) holds 2^-24 (sum of w n), row g8 + 8
            // (an odd nibble) 16 times that; 8 * (sum of w) is the offset of n = code + 8
            float b0 = 0.f, b1 = 0.f;
            if (f4) {
                float W0 = ws0, W1 = ws1;
#pragma unroll
                for (int off = 4; off < 32; off <<= 1) {
                    W0 += __shfl_xor_sync(0xffffffffu, W0, off);
                    W1 += __shfl_xor_sync(0xffffffffu, W1, off);
                }
                b0 = 8.f * W0;
                b1 = 8.f * W1;
            }
            const float ke = f4 ? 16777216.f : 1.f, ko = f4 ? 1048576.f : 1.f;  // 2^24, 2^20
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                // rows g8 and g8 + 8 of m-tile mt are channels dd and dd + 1 (4-bit: m-tile
                // mt covers channels 32 (mt / 2) + 4 g8 + 2 (mt % 2) + {0, 1}, see tile_i4)
                const int dd = f4 ? 32 * (mt >> 1) + 4 * g8 + 2 * (mt & 1) : mt * 16 + 2 * g8;
                // the lo parts of the weights' products: one query column, column 1
                // (g1_weights); a packed 4-bit piece, the lane gq/2 to the right (pv_i4)
                float x0 = o[mt][0], x1 = o[mt][1], x2 = o[mt][2], x3 = o[mt][3];
                if (p.gq == 1) {
                    x0 += x1;
                    x2 += x3;
                }
                if constexpr (PK) {
                    if (f4) {
                        const int src = lane + (p.gq >> 1);  // columns c + gq (tig < gq/2)
                        x0 += __shfl_sync(0xffffffffu, o[mt][0], src & 31);
                        x1 += __shfl_sync(0xffffffffu, o[mt][1], src & 31);
                        x2 += __shfl_sync(0xffffffffu, o[mt][2], src & 31);
                        x3 += __shfl_sync(0xffffffffu, o[mt][3], src & 31);
                    }
                }
                if (hA < p.gq)
                    *reinterpret_cast<float2*>(wo + hA * D + dd) =
                        make_float2((x0 * ke - b0) * rs, (x2 * ko - b0) * rs);
                if (hB < p.gq)
                    *reinterpret_cast<float2*>(wo + hB * D + dd) =
                        make_float2((x1 * ke - b1) * rs, (x3 * ko - b1) * rs);
            }
        }
    }
};

// The write half of the fused append: the new token of every (request, KV head) goes to its
// page and slot, and the open logical page's k_max / k_min take it in, exactly as
// dattn_kv_append writes one token (with a quantized pool, the row is quantized as that call
// quantizes it: the same row maximum, scale and codes). The work is spread over the consumer
// threads of all CTAs (one 8-channel chunk each; the chunks of a row are consecutive lanes).
// A CTA that reads the tile of a new token may see the slot before or after this write; it
// writes the new token into its stage itself (Consumer::patch_row, patch_row_q).
template <int D, int FMT>
__device__ void append_new_tokens(const AttnParams& p, const Smem& sm, int32_t cta, int32_t G,
                                  int ctid) {
    constexpr int VPR = D / 8;
    constexpr int NT = kConsumerWarps * 32;
    const int64_t n = (int64_t)p.B * p.Hkv * VPR;
    for (int64_t it = (int64_t)cta * NT + ctid; it < n; it += (int64_t)G * NT) {
        const int32_t c8 = (int32_t)(it % VPR);
        const int64_t bh = it / VPR;
        const int32_t b = (int32_t)(bh / p.Hkv), h = (int32_t)(bh - (int64_t)b * p.Hkv);
        const uint4 kv = __ldg(reinterpret_cast<const uint4*>(p.k_new + bh * D + c8 * 8));
        const uint4 vv = __ldg(reinterpret_cast<const uint4*>(p.v_new + bh * D + c8 * 8));
        float mk = 0.f, mv = 0.f;
        if constexpr (FMT != DATTN_KV_BF16) {
            // every lane of a row takes part in the row maxima, whatever its page; the lanes
            // in the loop are a prefix of the warp made of whole rows
            const int64_t warp_items = n - (it - (ctid & 31));
            const unsigned mask = warp_items >= 32 ? 0xffffffffu : ((1u << warp_items) - 1u);
            mk = row_absmax<VPR>(kv, mask);
            mv = row_absmax<VPR>(vv, mask);
        }
        const int32_t pos = sm.item_pos()[b];
        if (pos < 0) continue;  // flagged when the lengths were read
        const int32_t lp = pos / p.P;
        if (lp >= p.max_pages) {
            set_err(p.dev_err, DATTN_DEVERR_LEN_OOB);
            continue;
        }
        const int32_t page = __ldg(p.block_table + (int64_t)b * p.max_pages + lp);
        if (page < 0) {
            set_err(p.dev_err, DATTN_DEVERR_UNMAPPED_PAGE);
            continue;
        }
        if (page >= p.num_pages) {
            set_err(p.dev_err, DATTN_DEVERR_PAGE_OOB);
            continue;
        }
        const int32_t slot = pos - lp * p.P;
        const int64_t row = ((int64_t)page * p.Hkv + h) * p.P + slot;
        if constexpr (FMT == DATTN_KV_BF16) {
            const int64_t dst = (row * D + c8 * 8) * 2;
            *reinterpret_cast<uint4*>(p.k_pool_w + dst) = kv;
            *reinterpret_cast<uint4*>(p.v_pool_w + dst) = vv;
        } else {
            const bool i4 = FMT == DATTN_KV_INT4 || (FMT == DATTN_KV_MIXED && head_is_i4(p.hf, h));
            // the codes' row: the mixed pool keeps each format in its own region
            int64_t crow = row;
            uint8_t* kd = p.k_pool_w;
            uint8_t* vd = p.v_pool_w;
            if constexpr (FMT == DATTN_KV_MIXED) {
                const int32_t h4 = p.hf.h4, h8 = p.Hkv - h4;
                crow = ((int64_t)page * (i4 ? h4 : h8) + head_class_index(p.hf, h, i4)) * p.P +
                       slot;
                if (i4) {
                    const int64_t region8 = (int64_t)p.num_pages * h8 * p.P * D;
                    kd += region8;
                    vd += region8;
                }
            }
            float ks, vs;
            if (i4) {
                *reinterpret_cast<uint32_t*>(kd + crow * (D / 2) + c8 * 4) = quant4_chunk(kv, mk, ks);
                *reinterpret_cast<uint32_t*>(vd + crow * (D / 2) + c8 * 4) = quant4_chunk(vv, mv, vs);
            } else {
                *reinterpret_cast<uint2*>(kd + crow * D + c8 * 8) = quant8_chunk(kv, mk, ks);
                *reinterpret_cast<uint2*>(vd + crow * D + c8 * 8) = quant8_chunk(vv, mv, vs);
            }
            if (c8 == 0) {  // [row / 16][K, V][row % 16]
                float* sc = p.kv_scale_w + (row >> 4) * 32 + (row & 15);
                sc[0] = ks;
                sc[16] = vs;
            }
        }
        if (p.stats != nullptr) {
            uint16_t* st = p.stats +
                           (((int64_t)page * p.Hkv + h) * (p.P >> 4) + (slot >> 4)) * 2 * D + c8 * 8;
            uint4 mx = kv, mn = kv;  // a token at position % 16 == 0 opens its logical page
            if ((pos & 15) != 0) {
                mx = *reinterpret_cast<const uint4*>(st);
                mn = *reinterpret_cast<const uint4*>(st + D);
                bf16_fold8(kv, mx, mn);
            }
            *reinterpret_cast<uint4*>(st) = mx;
            *reinterpret_cast<uint4*>(st + D) = mn;
        }
    }
}

// Resident CTAs per SM the register budget is held to: three at d = 128, four at d = 64 and
// for the 4-bit pool, whose consumers bind it (96 registers; it fetches each piece's query at
// the piece's start instead of during the previous piece, which frees 16 of them).
template <int D, int FMT>
constexpr int attn_min_blocks() { return (D == 64 || FMT == DATTN_KV_INT4) ? 4 : 3; }

// APP: the launch of dattn_append_decode (the one-token append fused into the decode). It is
// a template parameter so that the plain decode carries none of the append's code and
// registers.
template <int D, int FMT, bool APP, bool PK>
__global__ void __launch_bounds__(kAttnThreads, attn_min_blocks<D, FMT>())
attention_kernel(const __grid_constant__ AttnParams p,
                 const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_v,
                 const __grid_constant__ CUtensorMap tmap_k4,
                 const __grid_constant__ CUtensorMap tmap_v4) {
    // tmap_k / tmap_v: the pool (the mixed pool: its 8-bit region); tmap_k4 / tmap_v4: the
    // mixed pool's 4-bit region (unused otherwise)
    extern __shared__ uint8_t smem_raw[];
    Smem sm;
    {  // align by the shared-window offset: the TMA swizzle pattern is defined on it
        const uint32_t off = smem_u32(smem_raw);
        sm.base = smem_raw + (((off + 1023u) & ~1023u) - off);
    }
    constexpr bool Q = FMT != DATTN_KV_BF16;  // a quantized pool with row scales
    sm.L = attn_smem_layout(D, p.gq, p.nitems, p.Hkv, p.mode == MODE_SPARSE, FMT, APP);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t G = gridDim.x, cta = blockIdx.x;
    constexpr int NS = attn_stages(FMT);

    // ---------------------------------------------------------------- setup
    // Before the dependency wait: only state that no kernel of this library writes.
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(sm.full_bar(s), 1);
            mbar_init(sm.empty_bar(s), 1);
        }
        *sm.abort_flag() = 0;
        fence_mbar_init();
    }
    if (warp == kConsumerWarps && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
        if constexpr (FMT == DATTN_KV_MIXED) {
            prefetch_tmap(&tmap_k4);
            prefetch_tmap(&tmap_v4);
        }
    }
    if (p.mode == MODE_SPARSE) {
        for (int h = tid; h < p.Hkv; h += kAttnThreads) {
            const int k = p.head_kind[h];
            sm.kinds()[h] = (k < 0 || k > 2) ? DATTN_HEAD_DENSE : k;
        }
        __syncthreads();
        if (tid == 0) {
            int32_t c0 = 0, c1 = 0, c2 = 0;
            for (int h = 0; h < p.Hkv; ++h) {
                int32_t* kb = sm.kind_before() + 3 * h;
                kb[0] = c0; kb[1] = c1; kb[2] = c2;
                const int k = sm.kinds()[h];
                c0 += k == DATTN_HEAD_DENSE;
                c1 += k == DATTN_HEAD_RETRIEVAL;
                c2 += k == DATTN_HEAD_STREAMING;
            }
            int32_t* kb = sm.kind_before() + 3 * p.Hkv;
            kb[0] = c0; kb[1] = c1; kb[2] = c2;
            make_aligned_plan(p, sm, G);
        }
    }
    {  // warm L2 with the metadata read right after the wait (each line by one thread)
        constexpr size_t kPrefetchCap = 16u << 20;
        const int64_t gt = (int64_t)cta * kAttnThreads + tid, gn = (int64_t)G * kAttnThreads;
        prefetch_l2_range(p.seq_lens, (size_t)p.B * 4u, gt, gn);
        const size_t bt_bytes = (size_t)p.B * p.max_pages * 4u;
        if (bt_bytes <= kPrefetchCap) prefetch_l2_range(p.block_table, bt_bytes, gt, gn);
        prefetch_l2_range(p.q, (size_t)p.B * p.Hq * D * 2u, gt, gn);
        if (p.mode == MODE_SPARSE && p.selected)
            prefetch_l2_range(p.selected, (size_t)p.B * p.Hkv * p.top_k * 4u, gt, gn);
        if (p.mode == MODE_SPARSE && p.selected_phys)
            prefetch_l2_range(p.selected_phys, (size_t)p.B * p.Hkv * p.top_k * 4u, gt, gn);
        if constexpr (APP) {
            prefetch_l2_range(p.k_new, (size_t)p.B * p.Hkv * D * 2u, gt, gn);
            prefetch_l2_range(p.v_new, (size_t)p.B * p.Hkv * D * 2u, gt, gn);
        }
        if (p.mode == MODE_PARTIAL) {
            prefetch_l2_range(p.chunk_req, (size_t)p.C * 4u, gt, gn);
            prefetch_l2_range(p.chunk_indptr, (size_t)(p.C + 1) * 4u, gt, gn);
        }
    }
    // From here on the lengths, the selection and the pool may come from the previous kernel.
    grid_dependency_wait();
    grid_launch_dependents();
    __syncthreads();
    const bool aligned = p.mode == MODE_SPARSE && sm.aplan()[AP_ON] != 0;
    // The lengths: with the fused append, request i attends one more token than seq_lens[i]
    // holds (its new token at position seq_lens[i]), as dattn_kv_append would leave it.
    auto length_of = [&](int32_t i) {
        int32_t L = p.seq_lens[i];
        const int32_t cap = p.max_pages * p.P;
        if constexpr (APP) {
            sm.item_pos()[i] = L;
            if (L >= 0 && L < cap) ++L;
        }
        if (L < 0 || L > cap) {
            set_err(p.dev_err, DATTN_DEVERR_LEN_OOB);
            L = min(max(L, 0), cap);
        }
        return L;
    };
    if (aligned) {
        for (int32_t i = tid; i < p.nitems; i += kAttnThreads) sm.item_len()[i] = length_of(i);
        __syncthreads();
    } else {
        // per-item costs, then an exclusive scan into item_start
        int32_t* st = sm.item_start();
        int32_t* ln = sm.item_len();
        const int32_t n = p.nitems;
        const int32_t per = (n + kAttnThreads - 1) / kAttnThreads;
        const int32_t i0 = min(n, tid * per), i1 = min(n, i0 + per);
        int32_t local_sum = 0;
        for (int32_t i = i0; i < i1; ++i) {
            int32_t cnt;
            if (p.mode == MODE_PARTIAL) {
                const int32_t b = p.chunk_req[i];
                const int32_t c0 = p.chunk_indptr[i], c1 = p.chunk_indptr[i + 1];
                int32_t npg = c1 - c0;
                // the chunk's page list must lie inside chunk_pages[0, chunk_indptr[C])
                if (b < 0 || b >= p.B || c0 < 0 || c1 > p.chunk_indptr[p.C] || npg < 0 ||
                    npg > p.max_pages) {
                    set_err(p.dev_err, DATTN_DEVERR_CHUNK_OOB);
                    npg = 0;
                }
                ln[i] = npg * (p.P >> 4);  // real tiles per head
                cnt = p.Hkv * Plan::cost_of(ln[i]);
            } else {
                const int32_t L = length_of(i);
                ln[i] = L;
                if (p.mode == MODE_SPARSE) {
                    const int32_t* kb = sm.kind_before() + 3 * p.Hkv;
                    cnt = kb[0] * Plan::cost_of(head_tiles(DATTN_HEAD_DENSE, L, p)) +
                          kb[1] * Plan::cost_of(head_tiles(DATTN_HEAD_RETRIEVAL, L, p)) +
                          kb[2] * Plan::cost_of(head_tiles(DATTN_HEAD_STREAMING, L, p));
                } else {
                    cnt = p.Hkv * Plan::cost_of(ceil16(L));
                }
            }
            local_sum += cnt;
            st[i] = cnt;  // each thread converts only its own entries below
        }
        // block-wide exclusive scan of the per-thread sums (threads own contiguous items)
        int32_t incl = local_sum;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t v = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += v;
        }
        if (lane == 31) sm.scan()[warp] = incl;
        __syncthreads();
        int32_t run = incl - local_sum;
        for (int w = 0; w < warp; ++w) run += sm.scan()[w];
        for (int32_t i = i0; i < i1; ++i) {
            const int32_t c = st[i];
            st[i] = run;
            run += c;
        }
        if (tid == 0) {
            int32_t tot = 0;
            for (int w = 0; w < kAttnThreads / 32; ++w) tot += sm.scan()[w];
            st[n] = tot;
        }
        __syncthreads();
    }
    const Plan plan(p, sm);
    int32_t W = 0, Gw = 1, X0 = 0, X1 = 0;
    if (!aligned) {
        W = sm.item_start()[p.nitems];
        // Only the first min(G, W) CTAs take work, so that every participating CTA owns at
        // least one cost unit. A CTA strictly between the first and the last owner of a
        // segment's real tiles lies inside them, so the pieces of a segment come from
        // consecutive CTAs c_first..c_last, each of which arrives on its counter once.
        Gw = W < G ? (W > 0 ? W : 1) : G;
        X0 = cta < Gw ? (int32_t)split_begin(W, Gw, cta) : 0;
        X1 = cta < Gw ? (int32_t)split_begin(W, Gw, cta + 1) : 0;
        // segments without tiles have no owner: CTA (s mod G) writes their empty result
        for (int32_t s = cta; s < p.nseg; s += G) {
            int32_t st, real, cost;
            plan.seg_span(s, st, real, cost);
            if (real == 0) {
                for (int idx = tid; idx < p.gq * D; idx += kAttnThreads)
                    write_final(p, s, idx / D, idx % D, D, kNegInf, 0.f, 0.f);
            }
        }
    }
    if (tid == 0) {
        int32_t* cp = sm.cplan();
        cp[0] = aligned ? 1 : 0;
        cp[1] = W;
        cp[2] = Gw;
        cp[3] = X0;
        cp[4] = X1;
    }
    __syncthreads();
    const PieceIter pieces(p, sm, plan, cta);
    int32_t cur0 = pieces.start();
    Piece first;
    const bool any = pieces.piece(cur0, first);

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer warp
        if (!any) return;
        const uint64_t pol = policy_evict_first();
        const uint32_t tile_bytes = attn_tile_bytes(FMT, D);
        const uint32_t tx = 2u * tile_bytes + (Q ? 128u : 0u);  // + the tile's 32 scales
        const uint32_t stages0 = smem_u32(sm.base + sm.L.stages);
        int32_t k = 0;  // real tiles issued so far: tile k uses stage k % NS
        bool stop = false;
        // Issues the nb tiles of this warp's batch (lane j resolved tile k + j into ref).
        // Returns false after an abort.
        auto issue = [&](const TileRef& ref, int32_t nb) -> bool {
            // Tiles go out kIssue at a time, lane j of a group taking tile k + j: it waits
            // for its stage to be released, posts the tile's token range, arms the full
            // barrier and issues the tile's copies (K and V boxes; with the 8-bit pool
            // also the run of 16 K and 16 V row scales).
            for (int32_t j0 = 0; j0 < nb; j0 += kIssue) {
                const int32_t n = min(kIssue, nb - j0);
                const int32_t src = min(j0 + lane, 31);
                const int32_t y = __shfl_sync(0xffffffffu, ref.y, src);
                const int32_t lohi = __shfl_sync(0xffffffffu, ref.lohi, src);
                int32_t yc = y;
                if constexpr (FMT == DATTN_KV_MIXED) yc = __shfl_sync(0xffffffffu, ref.yc, src);
                bool ok = true;
                if (lane < n) {
                    const int32_t kk = k + lane;
                    const int stg = kk % NS;
                    if (kk >= NS)
                        ok = mbar_wait(sm.empty_bar(stg), ((kk / NS) - 1) & 1,
                                       sm.abort_flag(), p.dev_err);
                    if (ok) {
                        const uint32_t full = sm.full_bar(stg);
                        sm.meta()[stg] = lohi;
                        if (lohi & kTileSkip) {
                            mbar_arrive(full);
                        } else if constexpr (FMT == DATTN_KV_MIXED) {
                            // a 4-bit tile takes the first half of the 8-bit stage: K codes,
                            // then V codes at 8 d bytes, where the 4-bit consumer reads them
                            const bool f4 = (lohi & kTileI4) != 0;
                            const uint32_t tb = f4 ? tile_bytes / 2u : tile_bytes;
                            mbar_arrive_expect_tx(full, 2u * tb + 128u);
                            const uint32_t dst = stages0 + (uint32_t)stg * sm.L.stage_bytes;
                            tma_load_2d(dst, f4 ? &tmap_k4 : &tmap_k, 0, yc, full, pol);
                            tma_load_2d(dst + tb, f4 ? &tmap_v4 : &tmap_v, 0, yc, full, pol);
                            bulk_copy(smem_u32(sm.scales(stg)), p.kv_scale + 2 * y, 128u, full,
                                      pol);
                        } else {
                            mbar_arrive_expect_tx(full, tx);
                            const uint32_t dst = stages0 + (uint32_t)stg * sm.L.stage_bytes;
                            if constexpr (Q) {
                                tma_load_2d(dst, &tmap_k, 0, y, full, pol);
                                tma_load_2d(dst + tile_bytes, &tmap_v, 0, y, full, pol);
                                // the tile's scales: 128 bytes at tile index y / 16
                                bulk_copy(smem_u32(sm.scales(stg)), p.kv_scale + 2 * y, 128u,
                                          full, pol);
                            } else {
                                tma_load_3d(dst, &tmap_k, 0, y, 0, full, pol);
                                tma_load_3d(dst + tile_bytes, &tmap_v, 0, y, 0, full, pol);
                            }
                        }
                    }
                }
                k += n;
                if (__any_sync(0xffffffffu, !ok)) return false;
            }
            return true;
        };
        {
            int32_t cur = cur0;
            Piece pc = first;
            int32_t base = pc.r0;
            bool have = true;
            while (have && !stop) {
                // Lanes take the next (up to) 32 tiles of the CTA's sequence, across piece
                // boundaries, so that the lookups of many small pieces overlap.
                int32_t my_s = -1, my_local = 0, nb = 0;
                while (have && nb < 32) {
                    const int32_t n = min(32 - nb, pc.r1 - base);
                    if (lane >= nb && lane < nb + n) {
                        my_s = pc.s;
                        my_local = base + (lane - nb);
                    }
                    nb += n;
                    base += n;
                    if (base == pc.r1) {
                        pieces.advance(cur);
                        have = pieces.piece(cur, pc);
                        if (have) base = pc.r0;
                    }
                }
                TileRef ref{0, kTileSkip, 0};
                if (my_s >= 0) ref = resolve_tile(p, sm, my_s, my_local, pieces.aligned());
                stop = !issue(ref, nb);
            }
        }
        // after an abort, wait (bounded in total) for copies still in flight before the CTA
        // exits; stages whose tiles were never issued simply run into the deadline
        if (lane == 0 && *sm.abort_flag()) {
            const unsigned long long t0 = global_timer_ns();
            for (int32_t kk = max(0, k - NS); kk < k; ++kk) {
                while (!mbar_try_wait(sm.full_bar(kk % NS), (kk / NS) & 1) &&
                       global_timer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumer warps
    {
        if constexpr (APP) {
            // Every thread of this CTA has read the lengths (the barrier above). The CTA that
            // arrives last advances seq_lens, as dattn_kv_append does; no CTA waits for another.
            if (warp == 0) {
                int32_t last = 0;
                if (lane == 0) {
                    const int32_t prev = atom_add_acq_rel_gpu(p.counters + p.nseg, 1);
                    last = prev == G - 1;
                    if (last) p.counters[p.nseg] = 0;  // ready for the next launch
                }
                if (__shfl_sync(0xffffffffu, last, 0)) {
                    for (int32_t i = lane; i < p.B; i += 32) {
                        const int32_t L = p.seq_lens_w[i];
                        if (L >= 0 && L < 0x7fffffff) p.seq_lens_w[i] = L + 1;
                    }
                }
            }
            append_new_tokens<D, FMT>(p, sm, cta, G, tid);
        }
    }
    if (!any) return;
    Consumer<D, FMT, PK> cons(p, sm, warp, lane);
    const uint32_t stage0 = smem_u32(sm.base + sm.L.stages);
    int32_t kbase = 0;  // real tiles of earlier pieces
    int32_t cur = cur0;
    Piece pc = first;
    bool have = true;
    uint32_t qn[Consumer<D, FMT, PK>::KS][2];
    float qsn = 0.f;
    // the 4-bit pool fetches each piece's query at its start (registers for four CTAs per SM)
    constexpr bool kPrefetchQ = FMT != DATTN_KV_INT4;
    float qcn[2] = {0.f, 0.f};
    if constexpr (kPrefetchQ) cons.load_q(pc.s, qn, qsn, qcn);
    while (have) {
        if constexpr (kPrefetchQ) {
#pragma unroll
            for (int ks = 0; ks < Consumer<D, FMT, PK>::KS; ++ks) {
                cons.qf[ks][0] = qn[ks][0];
                cons.qf[ks][1] = qn[ks][1];
            }
            cons.qsc = qsn;
            cons.qc[0] = qcn[0];
            cons.qc[1] = qcn[1];
        } else {
            cons.load_q(pc.s, cons.qf, cons.qsc, cons.qc);
        }
        // the next piece's query is fetched while this piece streams (only its cursor stays
        // live; the piece is looked up again at the switch)
        int32_t cur2 = cur;
        pieces.advance(cur2);
        bool have2;
        {
            Piece nx;
            have2 = pieces.piece(cur2, nx);
            if (kPrefetchQ && have2) cons.load_q(nx.s, qn, qsn, qcn);
        }
        // with the fused append, this lane's chunk of the segment's new K / V row (the tile
        // that holds the new token gets it written into its row)
        uint4 patch = make_uint4(0u, 0u, 0u, 0u);
        if constexpr (FMT == DATTN_KV_BF16) {
            if constexpr (APP) patch = cons.load_new_row(pc.s);
        }
        cons.reset();
        if constexpr (FMT == DATTN_KV_MIXED) cons.i4 = head_is_i4(p.hf, pc.s % p.Hkv);
        if constexpr (Consumer<D, FMT, PK>::Q) {
            if constexpr (APP) cons.quant_new_row(pc.s, Consumer<D, FMT, PK>::I4 || cons.i4);
        }
        const int32_t s = pc.s;
        const int32_t nr = pc.r1 - pc.r0;
        for (int32_t i = (warp - kbase % kConsumerWarps + kConsumerWarps) % kConsumerWarps;
             i < nr; i += kConsumerWarps) {
            const int32_t k = kbase + i;
            const int stg = k % NS;
            // warp-uniform: the tile's ldmatrix / mma / movmatrix are warp-collective
            const bool ok = __all_sync(0xffffffffu, mbar_wait(sm.full_bar(stg), (k / NS) & 1,
                                                              sm.abort_flag(), p.dev_err));
            const int32_t lohi = sm.meta()[stg];
            const int lo = tile_lo(lohi), hi = tile_hi(lohi), cut = tile_cut(lohi);
            if (ok && !(lohi & kTileSkip)) {
                if constexpr (Q) {
                    const uint32_t st = stage0 + (uint32_t)stg * sm.L.stage_bytes;
                    const bool t4 = FMT == DATTN_KV_INT4 ||
                                    (FMT == DATTN_KV_MIXED && (lohi & kTileI4) != 0);
                    // fused append: the new token's codes and scales into this stage, quantized
                    // here exactly as the write half quantizes them (the warp's lanes together)
                    const bool patched = APP && (lohi & kTilePatch) != 0;
                    if (patched)
                        cons.store_row_q(st, const_cast<float*>(sm.scales(stg)),
                                         tile_patch_row(lohi), t4);
                    if (t4) cons.tile_i4(st, sm.scales(stg), lo, hi, cut);
                    else    cons.tile_f8(st, sm.scales(stg), lo, hi, cut);
                    // generic writes to the stage before TMA refills it
                    if (patched) fence_proxy_async_smem();
                } else {
                    const uint32_t st = stage0 + (uint32_t)stg * sm.L.stage_bytes;
                    const bool patched = APP && (lohi & kTilePatch) != 0;
                    if (patched) cons.patch_row(st, tile_patch_row(lohi), patch);
                    cons.tile(st, lo, hi, cut);
                    // generic writes to the stage (patch, zeroed rows) before TMA refills it
                    if (patched || lo > 0 || hi < 16) fence_proxy_async_smem();
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.empty_bar(stg));
        }
        kbase += nr;
        // ---- merge the four warps' states of this piece -------------------------------
        cons.publish();
        named_bar_sync(1, kConsumerWarps * 32);
        const int32_t c_first = pc.cfirst;
        const int32_t c_last = pc.clast;
        const bool whole = c_first == c_last;
        const int ctid = tid;  // 0..127
        constexpr int kCT = kConsumerWarps * 32;
        const float* wm = sm.ws_m();
        const float* we = sm.ws_e();
        const float* wo = sm.ws_o();
        const int gD = p.gq * D;
        const int32_t slot_stride = slot_floats(p.gq, D);
        float* my_slot = whole ? nullptr : p.slots + (int64_t)(cta + s) * slot_stride;
        // a thread combines float4 columns of the g x D state; D is a multiple of 4, so a
        // column never spans two heads
        for (int c4 = ctid; c4 < gD / 4; c4 += kCT) {
            const int j = (4 * c4) / D, d = 4 * c4 - j * D;
            float mc = kNegInf;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) mc = fmaxf(mc, wm[w * kMaxGroup + j]);
            float ec = 0.f;
            float4 ma = make_float4(0.f, 0.f, 0.f, 0.f);
            if (mc != kNegInf) {
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const float mw = wm[w * kMaxGroup + j];
                    if (mw == kNegInf) continue;
                    const float sc = exp2f(mw - mc);
                    ec += we[w * kMaxGroup + j] * sc;
                    const float4 v = *reinterpret_cast<const float4*>(wo + w * gD + 4 * c4);
                    ma.x += v.x * sc;
                    ma.y += v.y * sc;
                    ma.z += v.z * sc;
                    ma.w += v.w * sc;
                }
            }
            if (whole) {
                write_final(p, s, j, d, D, mc, ec, ma.x);
                write_final(p, s, j, d + 1, D, mc, ec, ma.y);
                write_final(p, s, j, d + 2, D, mc, ec, ma.z);
                write_final(p, s, j, d + 3, D, mc, ec, ma.w);
            } else {
                *reinterpret_cast<float4*>(my_slot + 4 * c4) = ma;
                if (d == 0) {
                    my_slot[gD + j] = mc;
                    my_slot[gD + p.gq + j] = ec;
                }
            }
        }
        if (!whole) {
            // hand the piece over: the CTA that delivers the last piece merges them all
            named_bar_sync(1, kCT);
            const int32_t npieces = c_last - c_first + 1;
            if (ctid == 0) {
                // release: this CTA's slot writes (ordered before by the barrier) become
                // visible before the count; acquire: the last arrival sees every slot
                const int32_t prev = atom_add_acq_rel_gpu(p.counters + s, 1);
                *sm.last_flag() = (prev == npieces - 1) ? 1 : 0;
                if (prev == npieces - 1) p.counters[s] = 0;  // ready for the next launch
            }
            named_bar_sync(1, kCT);
            if (*sm.last_flag()) {
                // Merge all pieces of the segment. Each thread owns float4 columns of one
                // head's MA; for up to kMergeBatch pieces at a time it loads the pieces' (m, e)
                // of that head and its MA columns together, then folds them into a running
                // max, sum and accumulator (the weights are recomputed per thread).
                const float* first = p.slots + (int64_t)(c_first + s) * slot_stride;
                constexpr int kMergeBatch = 8;
                for (int c4 = ctid; c4 < gD / 4; c4 += kCT) {
                    const int j = (4 * c4) / D, d = 4 * c4 - j * D;
                    float mrun = kNegInf, erun = 0.f;
                    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int32_t q0 = 0; q0 < npieces; q0 += kMergeBatch) {
                        const float* pass = first + (int64_t)q0 * slot_stride;
                        float mq[kMergeBatch], eq[kMergeBatch];
                        float4 vq[kMergeBatch];
#pragma unroll
                        for (int t = 0; t < kMergeBatch; ++t) {
                            const bool in = q0 + t < npieces;
                            const float* sl = pass + (int64_t)t * slot_stride;
                            mq[t] = in ? __ldcg(sl + gD + j) : kNegInf;
                            eq[t] = in ? __ldcg(sl + gD + p.gq + j) : 0.f;
                            vq[t] = in ? __ldcg(reinterpret_cast<const float4*>(sl + 4 * c4))
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
                        float mx = mrun;
#pragma unroll
                        for (int t = 0; t < kMergeBatch; ++t) mx = fmaxf(mx, mq[t]);
                        if (mx == kNegInf) continue;  // every piece so far is empty
                        const float al = mrun == kNegInf ? 0.f : exp2f(mrun - mx);
                        erun *= al;
                        acc.x *= al;
                        acc.y *= al;
                        acc.z *= al;
                        acc.w *= al;
#pragma unroll
                        for (int t = 0; t < kMergeBatch; ++t) {
                            const float w = mq[t] == kNegInf ? 0.f : exp2f(mq[t] - mx);
                            erun += eq[t] * w;
                            acc.x += w * vq[t].x;
                            acc.y += w * vq[t].y;
                            acc.z += w * vq[t].z;
                            acc.w += w * vq[t].w;
                        }
                        mrun = mx;
                    }
                    write_final(p, s, j, d, D, mrun, erun, acc.x);
                    write_final(p, s, j, d + 1, D, mrun, erun, acc.y);
                    write_final(p, s, j, d + 2, D, mrun, erun, acc.z);
                    write_final(p, s, j, d + 3, D, mrun, erun, acc.w);
                }
            }
        }
        named_bar_sync(1, kConsumerWarps * 32);  // shared state is reused by the next piece
        cur = cur2;
        have = have2 && pieces.piece(cur, pc);
    }
}

// ------------------------------------------------------------------ host side
struct KernelInfo {
    int max_smem_set = 0;
};

template <int D, int FMT, bool APP, bool PK>
KernelInfo& kernel_info() {
    static KernelInfo info;
    return info;
}

std::mutex g_attr_mutex;

template <int D, int FMT, bool APP, bool PK>
dattn_status_t ensure_smem(uint32_t bytes) {
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    KernelInfo& ki = kernel_info<D, FMT, APP, PK>();
    if ((int)bytes > ki.max_smem_set) {
        if (cudaFuncSetAttribute(attention_kernel<D, FMT, APP, PK>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)bytes) != cudaSuccess)
            return DATTN_ERR_CUDA;
        ki.max_smem_set = (int)bytes;
    }
    return DATTN_OK;
}

template <int D, int FMT, bool APP, bool PK>
int occupancy(uint32_t smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attention_kernel<D, FMT, APP, PK>, kAttnThreads,
                                                      smem) != cudaSuccess)
        return 1;
    return n < 1 ? 1 : n;
}

}  // namespace

size_t attn_workspace_bytes(int32_t nseg, int32_t g, int32_t D, int32_t G) {
    return attn_counter_bytes(nseg) + (size_t)(G + nseg) * slot_floats(g, D) * 4;
}


template <int D, int FMT, bool APP, bool PK>
static dattn_status_t launch_d(const AttnParams& p0, const void* k_pool, const void* v_pool,
                               int32_t num_splits, void* ws, size_t ws_bytes,
                               cudaStream_t stream, int64_t tiles_bound) {
    AttnParams p = p0;
    const AttnSmem L =
        attn_smem_layout(D, p.gq, p.nitems, p.Hkv, p.mode == MODE_SPARSE, FMT, APP);
    dattn_status_t st = ensure_smem<D, FMT, APP, PK>(L.total);
    if (st != DATTN_OK) return st;
    const int32_t G = choose_splits(tiles_bound, num_splits, occupancy<D, FMT, APP, PK>(L.total));
    const size_t counters = attn_counter_bytes(p.nseg);
    if (ws == nullptr || ws_bytes < attn_workspace_bytes(p.nseg, p.gq, D, G) ||
        (reinterpret_cast<uintptr_t>(ws) & 255))
        return DATTN_ERR_WORKSPACE;
    p.counters = static_cast<int32_t*>(ws);
    p.slots = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + counters);
    alignas(64) CUtensorMap tk;
    alignas(64) CUtensorMap tv;
    alignas(64) CUtensorMap tk4;
    alignas(64) CUtensorMap tv4;
    const int64_t rows = (int64_t)p.num_pages * p.Hkv * p.P;
    if constexpr (FMT == DATTN_KV_BF16) {
        if ((st = make_kv_tensor_map(&tk, k_pool, rows, D)) != DATTN_OK) return st;
        if ((st = make_kv_tensor_map(&tv, v_pool, rows, D)) != DATTN_OK) return st;
    } else if constexpr (FMT == DATTN_KV_MIXED) {
        // the 8-bit region [num_pages][H8][P][d], then the 4-bit region [num_pages][H4][P][d/2];
        // a format without heads gets the other region's map (no tile uses it)
        const int64_t rows8 = (int64_t)p.num_pages * (p.Hkv - p.hf.h4) * p.P;
        const int64_t rows4 = (int64_t)p.num_pages * p.hf.h4 * p.P;
        const uint8_t* k4 = static_cast<const uint8_t*>(k_pool) + rows8 * D;
        const uint8_t* v4 = static_cast<const uint8_t*>(v_pool) + rows8 * D;
        if (rows4 > 0) {
            if ((st = make_kv_tensor_map_u8(&tk4, k4, rows4, D / 2)) != DATTN_OK) return st;
            if ((st = make_kv_tensor_map_u8(&tv4, v4, rows4, D / 2)) != DATTN_OK) return st;
        }
        if (rows8 > 0) {
            if ((st = make_kv_tensor_map_u8(&tk, k_pool, rows8, D)) != DATTN_OK) return st;
            if ((st = make_kv_tensor_map_u8(&tv, v_pool, rows8, D)) != DATTN_OK) return st;
        }
        if (rows4 == 0) tk4 = tk, tv4 = tv;
        if (rows8 == 0) tk = tk4, tv = tv4;
    } else {
        const int row_bytes = FMT == DATTN_KV_INT4 ? D / 2 : D;
        if ((st = make_kv_tensor_map_u8(&tk, k_pool, rows, row_bytes)) != DATTN_OK) return st;
        if ((st = make_kv_tensor_map_u8(&tv, v_pool, rows, row_bytes)) != DATTN_OK) return st;
    }
    if constexpr (FMT != DATTN_KV_MIXED) tk4 = tk, tv4 = tv;  // not read
    if (launch_pdl(attention_kernel<D, FMT, APP, PK>, dim3(G), dim3(kAttnThreads), L.total, stream, p, tk,
                   tv, tk4, tv4) != cudaSuccess)
        return DATTN_ERR_CUDA;
    return DATTN_OK;
}

dattn_status_t launch_attention(const AttnParams& p, const void* k_pool, const void* v_pool,
                                int D, int32_t num_splits, void* ws, size_t ws_bytes,
                                cudaStream_t stream, int64_t tiles_bound) {
    if (D != 64 && D != 128) return DATTN_ERR_UNSUPPORTED;
    // 2 or 4 query columns over the 4-bit pool: the packed-column consumers. (The mixed pool's
    // 4-bit heads keep two products per m-tile: a packed instance of the mixed kernel slowed
    // its 8-bit tiles, 27.0 against 25.1 µs per sparse-512k launch.)
    const bool pk = p.fmt == DATTN_KV_INT4 && (p.gq == 2 || p.gq == 4);
    auto pick = [&](auto bf16, auto f8, auto i4, auto mix, auto i4p) {
        return p.fmt == DATTN_KV_MIXED    ? mix
             : p.fmt == DATTN_KV_INT4     ? (pk ? i4p : i4)
             : p.fmt == DATTN_KV_FP8_E4M3 ? f8
                                          : bf16;
    };
#define DATTN_LAUNCHES(D_, APP_)                                                                \
    pick(launch_d<D_, DATTN_KV_BF16, APP_, false>, launch_d<D_, DATTN_KV_FP8_E4M3, APP_, false>,  \
         launch_d<D_, DATTN_KV_INT4, APP_, false>, launch_d<D_, DATTN_KV_MIXED, APP_, false>,     \
         launch_d<D_, DATTN_KV_INT4, APP_, true>)
    auto launch = p.append != 0 ? (D == 64 ? DATTN_LAUNCHES(64, true) : DATTN_LAUNCHES(128, true))
                                : (D == 64 ? DATTN_LAUNCHES(64, false) : DATTN_LAUNCHES(128, false));
#undef DATTN_LAUNCHES
    return launch(p, k_pool, v_pool, num_splits, ws, ws_bytes, stream, tiles_bound);
}

}  // namespace dattn
