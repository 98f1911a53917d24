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
// streams 16-token K and V row groups into an 8-stage shared-memory ring with 2-D TMA
// tensor loads: 128-byte swizzle, evict-first L2 policy, completion on mbarriers. Four
// consumer warps each own every fourth stage. A consumer runs the small QK^T tile with
// tokens as the M dimension and the GQA group as N (mma.sync m16n8k16, bf16 in, fp32
// accumulate). It does an online softmax in base 2 with warp shuffles, transposes P with
// movmatrix, and accumulates O^T = V^T P^T with P split into two bf16 terms, so the weights
// keep 16 significant bits. The work of all (segment = request or chunk, KV head) pairs is
// laid end to end in 16-token tiles and cut into equal contiguous ranges, one per CTA. Each
// CTA therefore gets the same number of bytes, whatever the length mix. A segment that
// lies inside one CTA is finished there. A segment cut across CTAs leaves one partial
// triple per CTA in the workspace, and the CTA that arrives last (atomic counter) merges
// them. No CTA ever waits on another.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dattn {

namespace {

#define kNegInf (-__int_as_float(0x7f800000))

struct Smem {
    uint8_t* base;
    AttnSmem L;
    __device__ uint32_t full_bar(int s) const { return smem_u32(base + L.bars) + 8u * s; }
    __device__ uint32_t empty_bar(int s) const {
        return smem_u32(base + L.bars) + 8u * (kStages + s);
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
    __device__ int32_t* scan() const { return reinterpret_cast<int32_t*>(base + L.scan); }
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

// Segment geometry derived from the per-item prefix sums in shared memory.
struct Plan {
    const AttnParams& p;
    const Smem& sm;
    __device__ Plan(const AttnParams& p_, const Smem& sm_) : p(p_), sm(sm_) {}

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

    // Offset of head h's tiles within item i, and head h's tile count.
    __device__ void head_span(int32_t i, int32_t h, int32_t& off, int32_t& len) const {
        if (p.mode == MODE_SPARSE) {
            const int32_t L = sm.item_len()[i];
            const int32_t n0 = head_tiles(DATTN_HEAD_DENSE, L, p);
            const int32_t n1 = head_tiles(DATTN_HEAD_RETRIEVAL, L, p);
            const int32_t n2 = head_tiles(DATTN_HEAD_STREAMING, L, p);
            const int32_t* kb = sm.kind_before() + 3 * h;
            off = kb[0] * n0 + kb[1] * n1 + kb[2] * n2;
            const int k = sm.kinds()[h];
            len = k == DATTN_HEAD_RETRIEVAL ? n1 : (k == DATTN_HEAD_STREAMING ? n2 : n0);
        } else {
            const int32_t per = (sm.item_start()[i + 1] - sm.item_start()[i]) / p.Hkv;
            off = h * per;
            len = per;
        }
    }

    __device__ void seg_span(int32_t s, int32_t& start, int32_t& len) const {
        const int32_t i = s / p.Hkv, h = s - i * p.Hkv;
        int32_t off;
        head_span(i, h, off, len);
        start = sm.item_start()[i] + off;
    }

    // Segment containing tile t, and t's index inside it.
    __device__ void locate(int32_t t, int32_t& s, int32_t& local) const {
        const int32_t i = item_of(t);
        const int32_t o = t - sm.item_start()[i];
        int32_t h;
        if (p.mode == MODE_SPARSE) {
            // largest head whose offset is <= o; its range is non-empty and contains o
            int32_t lo = 0, hi = p.Hkv - 1;
            while (lo < hi) {
                const int32_t mid = (lo + hi + 1) >> 1;
                int32_t off, len;
                head_span(i, mid, off, len);
                if (off <= o) lo = mid; else hi = mid - 1;
            }
            h = lo;
        } else {
            const int32_t per = (sm.item_start()[i + 1] - sm.item_start()[i]) / p.Hkv;
            h = o / per;
        }
        int32_t off, len;
        head_span(i, h, off, len);
        s = i * p.Hkv + h;
        local = o - off;
    }
};

// Resolved tile: TMA row coordinate and the valid token range [lo, hi) within its 16 rows.
struct TileRef {
    int32_t y;
    int32_t lohi;  // lo | hi << 8 | skip << 16
};

__device__ __forceinline__ TileRef resolve_tile(const AttnParams& p, const Smem& sm, int32_t s,
                                                int32_t local) {
    TileRef r{0, 1 << 16};
    const int32_t item = s / p.Hkv, h = s - item * p.Hkv;
    int32_t b, L, t0, lo = 0, hi = 16;
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
            const int32_t per_page = p.P >> 4;
            const int32_t si = local / per_page;
            const int32_t pg = __ldg(p.selected + ((int64_t)b * p.Hkv + h) * p.top_k + si);
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
            if (local < nsink) {
                t0 = local * 16;
                hi = min(16, s_end - t0);
            } else {
                t0 = ((l0 >> 4) + (local - nsink)) * 16;
                lo = max(t0, l0) - t0;
                hi = min(t0 + 16, L) - t0;
            }
        } else {
            t0 = local * 16;
            hi = min(16, L - t0);
        }
    }
    const int32_t lp = t0 / p.P;
    const int32_t page = __ldg(p.block_table + (int64_t)b * p.max_pages + lp);
    if (page < 0) {
        set_err(p.dev_err, DATTN_DEVERR_UNMAPPED_PAGE);
        return r;
    }
    if (page >= p.num_pages) {
        set_err(p.dev_err, DATTN_DEVERR_PAGE_OOB);
        return r;
    }
    r.y = (page * p.Hkv + h) * p.P + (t0 - lp * p.P);
    r.lohi = lo | (hi << 8);
    return r;
}

// Writes the final result of query heads [kvh*g, kvh*g + g) of segment s.
// MA is unnormalised; m is in log2 units.
__device__ __forceinline__ void write_final(const AttnParams& p, int32_t s, int32_t j, int32_t d,
                                            int D, float m, float e, float ma) {
    const int32_t item = s / p.Hkv, kvh = s - item * p.Hkv;
    const int64_t row = (int64_t)item * p.Hq + kvh * p.g + j;
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

template <int D>
struct Consumer {
    static constexpr int KS = D / 16;  // k-steps of QK^T and m-tiles of PV

    const AttnParams& p;
    const Smem& sm;
    const int warp, lane;
    uint32_t qf[KS][2];
    float o[KS][4];
    float m0, m1, e0, e1;

    __device__ Consumer(const AttnParams& p_, const Smem& sm_, int w, int l)
        : p(p_), sm(sm_), warp(w), lane(l) {}

    __device__ void load_q(int32_t s) {
        const int32_t item = s / p.Hkv, kvh = s - item * p.Hkv;
        int32_t b = item;
        if (p.mode == MODE_PARTIAL) b = __ldg(p.chunk_req + item);
        const int n = lane >> 2, tig = lane & 3;
        const bool ok = n < p.g && b >= 0 && b < p.B;
        const uint32_t* qv = reinterpret_cast<const uint32_t*>(
            p.q + ((int64_t)(ok ? b : 0) * p.Hq + kvh * p.g + (ok ? n : 0)) * D);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            qf[ks][0] = ok ? __ldg(qv + ks * 8 + tig) : 0u;
            qf[ks][1] = ok ? __ldg(qv + ks * 8 + 4 + tig) : 0u;
        }
    }

    __device__ void reset() {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
        m0 = m1 = kNegInf;
        e0 = e1 = 0.f;
    }

    // One 16-token tile in stage buffer `st`; rows outside [lo, hi) are masked.
    __device__ void tile(uint32_t st, int lo, int hi) {
        const uint32_t kbase = st, vbase = st + (uint32_t)(D / 64) * 2048u;
        const int g8 = lane >> 2;
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
        const bool v0 = g8 >= lo && g8 < hi, v1 = g8 + 8 >= lo && g8 + 8 < hi;
        const float s0 = v0 ? (sa[0] + sb[0]) * p.sl2 : kNegInf;
        const float s1 = v0 ? (sa[1] + sb[1]) * p.sl2 : kNegInf;
        const float s2 = v1 ? (sa[2] + sb[2]) * p.sl2 : kNegInf;
        const float s3 = v1 ? (sa[3] + sb[3]) * p.sl2 : kNegInf;
        // ---- online softmax (base 2) ------------------------------------------------
        float c0 = fmaxf(s0, s2), c1 = fmaxf(s1, s3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            c0 = fmaxf(c0, __shfl_xor_sync(0xffffffffu, c0, off));
            c1 = fmaxf(c1, __shfl_xor_sync(0xffffffffu, c1, off));
        }
        const float mn0 = fmaxf(m0, c0), mn1 = fmaxf(m1, c1);
        const float mu0 = mn0 == kNegInf ? 0.f : mn0, mu1 = mn1 == kNegInf ? 0.f : mn1;
        const float p0 = exp2f(s0 - mu0), p1 = exp2f(s1 - mu1);
        const float p2 = exp2f(s2 - mu0), p3 = exp2f(s3 - mu1);
        if (__any_sync(0xffffffffu, mn0 != m0 || mn1 != m1)) {
            const float al0 = exp2f(m0 - mu0), al1 = exp2f(m1 - mu1);
            e0 *= al0;
            e1 *= al1;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                o[mt][0] *= al0; o[mt][1] *= al1; o[mt][2] *= al0; o[mt][3] *= al1;
            }
        }
        m0 = mn0;
        m1 = mn1;
        e0 += p0 + p2;
        e1 += p1 + p3;
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
        float* wo = sm.ws_o() + warp * p.g * D;
        if (g8 == 0) {
            if (hA < p.g) { wm[hA] = m0; we[hA] = t0; }
            if (hB < p.g) { wm[hB] = m1; we[hB] = t1; }
        }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
            const int dd = mt * 16 + g8;
            if (hA < p.g) { wo[hA * D + dd] = o[mt][0]; wo[hA * D + dd + 8] = o[mt][2]; }
            if (hB < p.g) { wo[hB * D + dd] = o[mt][1]; wo[hB * D + dd + 8] = o[mt][3]; }
        }
    }
};

template <int D>
__global__ void __launch_bounds__(kAttnThreads)
attention_kernel(const __grid_constant__ AttnParams p,
                 const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_v) {
    extern __shared__ uint8_t smem_raw[];
    Smem sm;
    {  // align by the shared-window offset: the TMA swizzle pattern is defined on it
        const uint32_t off = smem_u32(smem_raw);
        sm.base = smem_raw + (((off + 1023u) & ~1023u) - off);
    }
    sm.L = attn_smem_layout(D, p.g, p.nitems, p.Hkv, p.mode == MODE_SPARSE);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t G = gridDim.x, cta = blockIdx.x;

    // ---------------------------------------------------------------- setup
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(sm.full_bar(s), 1);
            mbar_init(sm.empty_bar(s), 1);
        }
        *sm.abort_flag() = 0;
        fence_mbar_init();
    }
    if (warp == kConsumerWarps && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    if (p.mode == MODE_SPARSE && tid == 0) {
        int32_t cnt[3] = {0, 0, 0};
        for (int h = 0; h < p.Hkv; ++h) {
            int k = p.head_kind[h];
            if (k < 0 || k > 2) k = DATTN_HEAD_DENSE;
            int32_t* kb = sm.kind_before() + 3 * h;
            kb[0] = cnt[0]; kb[1] = cnt[1]; kb[2] = cnt[2];
            sm.kinds()[h] = k;
            ++cnt[k];
        }
        int32_t* kb = sm.kind_before() + 3 * p.Hkv;
        kb[0] = cnt[0]; kb[1] = cnt[1]; kb[2] = cnt[2];
    }
    __syncthreads();
    // per-item tile counts, then an exclusive scan into item_start
    {
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
                int32_t npg = p.chunk_indptr[i + 1] - p.chunk_indptr[i];
                if (b < 0 || b >= p.B || npg < 0 || npg > p.max_pages) {
                    set_err(p.dev_err, DATTN_DEVERR_CHUNK_OOB);
                    npg = 0;
                }
                ln[i] = 0;
                cnt = p.Hkv * npg * (p.P >> 4);
            } else {
                int32_t L = p.seq_lens[i];
                const int32_t cap = p.max_pages * p.P;
                if (L < 0 || L > cap) {
                    set_err(p.dev_err, DATTN_DEVERR_LEN_OOB);
                    L = min(max(L, 0), cap);
                }
                ln[i] = L;
                if (p.mode == MODE_SPARSE) {
                    const int32_t* kb = sm.kind_before() + 3 * p.Hkv;
                    cnt = kb[0] * head_tiles(DATTN_HEAD_DENSE, L, p) +
                          kb[1] * head_tiles(DATTN_HEAD_RETRIEVAL, L, p) +
                          kb[2] * head_tiles(DATTN_HEAD_STREAMING, L, p);
                } else {
                    cnt = p.Hkv * ceil16(L);
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
    const int32_t W = sm.item_start()[p.nitems];
    // Only the first min(G, W) CTAs take tiles, so that every participating CTA owns at
    // least one tile: the pieces of a segment then come from consecutive CTAs
    // c_first..c_last, and each of them arrives on the segment's counter exactly once.
    const int32_t Gw = W < G ? (W > 0 ? W : 1) : G;
    const int32_t t_begin = cta < Gw ? (int32_t)split_begin(W, Gw, cta) : 0;
    const int32_t t_end = cta < Gw ? (int32_t)split_begin(W, Gw, cta + 1) : 0;

    // segments without tiles have no owner: CTA (s mod G) writes their empty result
    for (int32_t s = cta; s < p.nseg; s += G) {
        int32_t st, len;
        plan.seg_span(s, st, len);
        if (len == 0) {
            for (int idx = tid; idx < p.g * D; idx += kAttnThreads)
                write_final(p, s, idx / D, idx % D, D, kNegInf, 0.f, 0.f);
        }
    }
    if (t_begin >= t_end) return;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer warp
        const uint64_t pol = policy_evict_first();
        const uint32_t tile_bytes = (uint32_t)(D / 64) * 2048u;
        const int32_t ntiles = t_end - t_begin;
        int32_t issued = 0;
        bool stop = false;
        for (int32_t base = 0; base < ntiles && !stop; base += 32) {
            TileRef ref{0, 1 << 16};
            if (base + lane < ntiles) {
                int32_t s, local;
                plan.locate(t_begin + base + lane, s, local);
                ref = resolve_tile(p, sm, s, local);
            }
            const int32_t nb = min(32, ntiles - base);
            for (int32_t j = 0; j < nb; ++j) {
                const int32_t y = __shfl_sync(0xffffffffu, ref.y, j);
                const int32_t lohi = __shfl_sync(0xffffffffu, ref.lohi, j);
                if (lane == 0) {
                    const int32_t k = base + j;
                    const int stg = k % kStages;
                    bool ok = true;
                    if (k >= kStages)
                        ok = mbar_wait(sm.empty_bar(stg), ((k / kStages) - 1) & 1,
                                       sm.abort_flag(), p.dev_err);
                    if (!ok) {
                        stop = true;
                    } else {
                        sm.meta()[stg] = lohi;
                        const uint32_t full = sm.full_bar(stg);
                        if (lohi >> 16) {
                            mbar_arrive(full);
                        } else {
                            const uint32_t dst = smem_u32(sm.base + sm.L.stages) +
                                                 (uint32_t)stg * sm.L.stage_bytes;
                            mbar_arrive_expect_tx(full, 2u * tile_bytes);
#pragma unroll
                            for (int hf = 0; hf < D / 64; ++hf)
                                tma_load_2d(dst + hf * 2048u, &tmap_k, hf * 64, y, full, pol);
#pragma unroll
                            for (int hf = 0; hf < D / 64; ++hf)
                                tma_load_2d(dst + tile_bytes + hf * 2048u, &tmap_v, hf * 64, y,
                                            full, pol);
                        }
                        issued = k + 1;
                    }
                }
                stop = __shfl_sync(0xffffffffu, stop ? 1 : 0, 0) != 0;
                if (stop) break;
            }
        }
        // after an abort, wait (bounded) for copies still in flight before the CTA exits
        if (lane == 0 && *sm.abort_flag()) {
            for (int32_t k = max(0, issued - kStages); k < issued; ++k) {
                const unsigned long long t0 = global_timer_ns();
                while (!mbar_try_wait(sm.full_bar(k % kStages), (k / kStages) & 1) &&
                       global_timer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumer warps
    Consumer<D> cons(p, sm, warp, lane);
    const uint32_t stage0 = smem_u32(sm.base + sm.L.stages);
    int32_t s = 0, dummy = 0;
    plan.locate(t_begin, s, dummy);
    int32_t a = t_begin;
    while (a < t_end) {
        int32_t sst, slen;
        plan.seg_span(s, sst, slen);
        while (sst + slen <= a) {
            ++s;
            plan.seg_span(s, sst, slen);
        }
        const int32_t pe = min(sst + slen, t_end);
        cons.load_q(s);
        cons.reset();
        const int32_t ka = a - t_begin, kb = pe - t_begin;
        for (int32_t k = ka + ((warp - ka % kConsumerWarps + kConsumerWarps) % kConsumerWarps);
             k < kb; k += kConsumerWarps) {
            const int stg = k % kStages;
            // warp-uniform: the tile's ldmatrix / mma / movmatrix are warp-collective
            const bool ok = __all_sync(0xffffffffu, mbar_wait(sm.full_bar(stg), (k / kStages) & 1,
                                                              sm.abort_flag(), p.dev_err));
            const int32_t lohi = sm.meta()[stg];
            const int lo = lohi & 0xff, hi = (lohi >> 8) & 0xff;
            if (ok && !(lohi >> 16)) {
                cons.tile(stage0 + (uint32_t)stg * sm.L.stage_bytes, lo, hi);
                if (lo > 0 || hi < 16) fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(sm.empty_bar(stg));
        }
        // ---- merge the four warps' states of this piece -------------------------------
        cons.publish();
        named_bar_sync(1, kConsumerWarps * 32);
        const bool whole = (a == sst) && (pe == sst + slen);
        const int ctid = tid;  // 0..127
        float* wm = sm.ws_m();
        float* we = sm.ws_e();
        float* wo = sm.ws_o();
        const int gD = p.g * D;
        const int32_t slot_stride = p.g * (D + 2);
        float* my_slot = whole ? nullptr : p.slots + (int64_t)(cta + s) * slot_stride;
        for (int idx = ctid; idx < gD; idx += kConsumerWarps * 32) {
            const int j = idx / D, d = idx - j * D;
            float mc = kNegInf;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) mc = fmaxf(mc, wm[w * kMaxGroup + j]);
            float ec = 0.f, ma = 0.f;
            if (mc != kNegInf) {
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const float mw = wm[w * kMaxGroup + j];
                    if (mw == kNegInf) continue;
                    const float sc = exp2f(mw - mc);
                    ec += we[w * kMaxGroup + j] * sc;
                    ma += wo[w * gD + j * D + d] * sc;
                }
            }
            if (whole) {
                write_final(p, s, j, d, D, mc, ec, ma);
            } else {
                my_slot[j * D + d] = ma;
                if (d == 0) {
                    my_slot[gD + j] = mc;
                    my_slot[gD + p.g + j] = ec;
                }
            }
        }
        if (!whole) {
            // hand the piece over: the CTA that delivers the last piece merges them all
            named_bar_sync(1, kConsumerWarps * 32);
            const int32_t c_first = split_owner(sst, W, Gw);
            const int32_t c_last = split_owner(sst + slen - 1, W, Gw);
            const int32_t npieces = c_last - c_first + 1;
            if (ctid == 0) {
                __threadfence();
                const int32_t prev = atomicAdd(p.counters + s, 1);
                *sm.last_flag() = (prev == npieces - 1) ? 1 : 0;
                if (prev == npieces - 1) p.counters[s] = 0;  // ready for the next launch
            }
            named_bar_sync(1, kConsumerWarps * 32);
            if (*sm.last_flag()) {
                __threadfence();
                const float* first = p.slots + (int64_t)(c_first + s) * slot_stride;
                for (int idx = ctid; idx < gD; idx += kConsumerWarps * 32) {
                    const int j = idx / D, d = idx - j * D;
                    float mc = kNegInf;
                    for (int32_t q = 0; q < npieces; ++q)
                        mc = fmaxf(mc, __ldcg(first + (int64_t)q * slot_stride + gD + j));
                    float ec = 0.f, ma = 0.f;
                    if (mc != kNegInf) {
                        for (int32_t q = 0; q < npieces; ++q) {
                            const float* sl = first + (int64_t)q * slot_stride;
                            const float mq = __ldcg(sl + gD + j);
                            if (mq == kNegInf) continue;
                            const float sc = exp2f(mq - mc);
                            ec += __ldcg(sl + gD + p.g + j) * sc;
                            ma += __ldcg(sl + j * D + d) * sc;
                        }
                    }
                    write_final(p, s, j, d, D, mc, ec, ma);
                }
            }
        }
        named_bar_sync(1, kConsumerWarps * 32);  // shared state is reused by the next piece
        a = pe;
    }
}

// ------------------------------------------------------------------ host side
struct KernelInfo {
    int max_smem_set = 0;
};

template <int D>
KernelInfo& kernel_info() {
    static KernelInfo info;
    return info;
}

std::mutex g_attr_mutex;

template <int D>
dattn_status_t ensure_smem(uint32_t bytes) {
    std::lock_guard<std::mutex> lock(g_attr_mutex);
    KernelInfo& ki = kernel_info<D>();
    if ((int)bytes > ki.max_smem_set) {
        if (cudaFuncSetAttribute(attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)bytes) != cudaSuccess)
            return DATTN_ERR_CUDA;
        ki.max_smem_set = (int)bytes;
    }
    return DATTN_OK;
}

template <int D>
int occupancy(uint32_t smem) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, attention_kernel<D>, kAttnThreads,
                                                      smem) != cudaSuccess)
        return 1;
    return n < 1 ? 1 : n;
}

}  // namespace

size_t attn_workspace_bytes(int32_t nseg, int32_t g, int32_t D, int32_t G) {
    const size_t counters = ((size_t)nseg * 4 + 255) & ~(size_t)255;
    return counters + (size_t)(G + nseg) * g * (D + 2) * 4;
}

template <int D>
static dattn_status_t launch_d(const AttnParams& p0, const void* k_pool, const void* v_pool,
                               int32_t num_splits, void* ws, size_t ws_bytes,
                               cudaStream_t stream, int64_t tiles_bound) {
    AttnParams p = p0;
    const AttnSmem L = attn_smem_layout(D, p.g, p.nitems, p.Hkv, p.mode == MODE_SPARSE);
    dattn_status_t st = ensure_smem<D>(L.total);
    if (st != DATTN_OK) return st;
    const int32_t G = choose_splits(tiles_bound, num_splits, occupancy<D>(L.total));
    const size_t counters = ((size_t)p.nseg * 4 + 255) & ~(size_t)255;
    if (ws == nullptr || ws_bytes < attn_workspace_bytes(p.nseg, p.g, D, G) ||
        (reinterpret_cast<uintptr_t>(ws) & 255))
        return DATTN_ERR_WORKSPACE;
    p.counters = static_cast<int32_t*>(ws);
    p.slots = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + counters);
    alignas(64) CUtensorMap tk;
    alignas(64) CUtensorMap tv;
    const int64_t rows = (int64_t)p.num_pages * p.Hkv * p.P;
    if ((st = make_kv_tensor_map(&tk, k_pool, rows, D)) != DATTN_OK) return st;
    if ((st = make_kv_tensor_map(&tv, v_pool, rows, D)) != DATTN_OK) return st;
    attention_kernel<D><<<G, kAttnThreads, L.total, stream>>>(p, tk, tv);
    return cudaGetLastError() == cudaSuccess ? DATTN_OK : DATTN_ERR_CUDA;
}

dattn_status_t launch_attention(const AttnParams& p, const void* k_pool, const void* v_pool,
                                int D, int32_t num_splits, void* ws, size_t ws_bytes,
                                cudaStream_t stream, int64_t tiles_bound) {
    if (D == 64) return launch_d<64>(p, k_pool, v_pool, num_splits, ws, ws_bytes, stream,
                                     tiles_bound);
    if (D == 128) return launch_d<128>(p, k_pool, v_pool, num_splits, ws, ws_bytes, stream,
                                       tiles_bound);
    return DATTN_ERR_UNSUPPORTED;
}

int32_t attention_occupancy(int D, int g, int nitems, int Hkv, bool sparse) {
    const AttnSmem L = attn_smem_layout(D, g, nitems, Hkv, sparse);
    if (D == 64) { if (ensure_smem<64>(L.total) != DATTN_OK) return 1; return occupancy<64>(L.total); }
    if (ensure_smem<128>(L.total) != DATTN_OK) return 1;
    return occupancy<128>(L.total);
}

}  // namespace dattn
