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
// the g heads, so one selection serves the whole group. The sum is accumulated in fp32,
// one fused multiply-add per channel in ascending channel order. For q_d >= 0 the larger
// product is q_d * kmax_d, otherwise q_d * kmin_d. This fixed arithmetic decides the
// selection.
//
// GB300 design. The statistics scan is HBM-bound: every reuse window it reads all k_max and
// k_min of the retrieval heads (512 B per logical page at d = 128), and it must score them
// at that speed. The physical pages of all retrieval (request, KV head) pairs are laid end
// to end and cut into equal contiguous ranges, one per CTA (one CTA per SM).
//  - No staging: eight warps read the statistics straight into registers with coalesced
//    16-byte loads, software-pipelined three groups deep. A logical page's 2*d values are
//    spread over d/16 lanes (16 channels each), so each lane keeps the query values of its
//    channels for four heads in registers for the whole piece.
//  - A lane runs its 16 channels as two chains (even and odd channels) of packed fp32x2
//    fused multiply-adds, four heads at once. The lanes of a logical page then combine
//    their partial sums with a fixed butterfly.
//  - Page maxima that beat the warp's running K-th key go to a per-warp candidate buffer.
//    The buffer is folded into the warp's top K by a warp-synchronous bitonic sort.
//  - At the end of a piece the eight warps' lists are merged. A head split across CTAs
//    leaves each CTA's top K in the workspace, and the CTA that arrives last merges them.
//
// Decision arithmetic (the selection is an integer decided by floating point, so it is
// fixed exactly, and the oracle repeats it). For head j, channels are taken in chunks of C
// (C = 16 for groups of up to 4 query heads, C = 8 otherwise). Within a chunk there are two
// fp32 accumulators, for even and odd channels, both starting at +0. Each channel adds, by
// fused multiply-add, first max(q,0)*kmax then min(q,0)*kmin; one of the two is an exact
// zero, so this adds exactly the product q*kmax or q*kmin that the score definition selects.
// A chunk's partial is even + odd. The partials are summed by a pairwise tree: adjacent
// chunks first, then pairs of pairs.
#include "common.cuh"
#include "internal.h"

namespace dattn {

namespace {

constexpr int kSelWarps = 8;
constexpr int kSelThreads = kSelWarps * 32;
constexpr int kSelBlockPages = 1024;  // pages whose block-table entries are staged at once

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
    int32_t* counters;
    uint64_t* slots;
    int32_t nseg;
    int32_t* dev_err;
};

__host__ __device__ inline int next_pow2(int x) {
    int n = 1;
    while (n < x) n <<= 1;
    return n;
}

struct SelSmem {
    uint32_t flags, bt, wbuf, sortbuf, ret_before, ret_heads, item_start, item_len, scan, total;
    int wn, sn;
};

__host__ __device__ inline SelSmem sel_smem_layout(int B, int Hkv, int K) {
    SelSmem s;
    s.wn = next_pow2(2 * K);                 // per-warp buffer: top K + candidates
    s.sn = next_pow2(kSelWarps * K);         // CTA buffer: the warps' lists, or pieces to fold
    uint32_t o = 0;
    s.flags = o;      o += 16u;
    s.bt = o;         o += kSelBlockPages * 4u;
    o = (o + 15u) & ~15u;
    s.wbuf = o;       o += (uint32_t)kSelWarps * s.wn * 8u;
    s.sortbuf = o;    o += (uint32_t)s.sn * 8u;
    s.ret_before = o; o += (uint32_t)(Hkv + 1) * 4u;
    s.ret_heads = o;  o += (uint32_t)Hkv * 4u;
    o = (o + 15u) & ~15u;
    s.item_start = o; o += (uint32_t)(B + 1) * 4u;
    s.item_len = o;   o += (uint32_t)B * 4u;
    o = (o + 15u) & ~15u;
    s.scan = o;       o += 8u * 4u;
    s.total = o + 128u;
    return s;
}

__device__ __forceinline__ uint64_t make_key(float score, int32_t page) {
    const uint32_t u = __float_as_uint(score + 0.0f);  // -0 becomes +0
    const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    return ((uint64_t)ord << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)page);
}

__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// acc = a * b + acc, two independent IEEE fp32 fused multiply-adds
__device__ __forceinline__ void fma_f32x2(uint64_t& acc, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

// 16-byte streaming load (read once: no L1 allocation, evict-first in L2)
__device__ __forceinline__ uint4 ldg_stream(const void* ptr, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr), "l"(pol));
    return v;
}

// Bitonic sort of buf[0..n) into descending order by nthreads threads (index tid); sync()
// separates the steps.
template <typename Sync>
__device__ __forceinline__ void bitonic_desc(uint64_t* buf, int n, int tid, int nthreads,
                                             Sync sync) {
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int idx = tid; idx < (n >> 1); idx += nthreads) {
                const int i = 2 * j * (idx / j) + (idx % j);
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

// D: head_dim; CPL: channels per lane (16 or 8); HG: query heads per lane (4 or 8).
template <int D, int CPL, int HG>
__global__ void __launch_bounds__(kSelThreads, 1)
page_select_kernel(const __grid_constant__ SelParams p) {
    constexpr int LPR = D / CPL;     // lanes per logical page (row)
    constexpr int RPW = 32 / LPR;    // rows per warp group
    constexpr int NLD = CPL / 8;     // 16-byte loads per lane for k_max (and for k_min)
    constexpr int NPAIR = CPL / 2;   // channel pairs per lane
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_off = smem_u32(smem_raw);
    uint8_t* base = smem_raw + (((raw_off + 127u) & ~127u) - raw_off);
    const int K = p.top_k;
    const SelSmem L = sel_smem_layout(p.B, p.Hkv, K);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t G = gridDim.x, cta = blockIdx.x;
    const int LPG = p.P >> 4;
    int* last_flag = reinterpret_cast<int*>(base + L.flags);
    int32_t* bt_blk = reinterpret_cast<int32_t*>(base + L.bt);
    uint64_t* sortbuf = reinterpret_cast<uint64_t*>(base + L.sortbuf);
    int32_t* ret_before = reinterpret_cast<int32_t*>(base + L.ret_before);
    int32_t* ret_heads = reinterpret_cast<int32_t*>(base + L.ret_heads);
    int32_t* item_start = reinterpret_cast<int32_t*>(base + L.item_start);
    int32_t* item_len = reinterpret_cast<int32_t*>(base + L.item_len);
    int32_t* scan = reinterpret_cast<int32_t*>(base + L.scan);

    grid_dependency_wait();  // lengths and statistics may come from the previous kernel
    grid_launch_dependents();
    // ---------------------------------------------------------------- setup
    for (int h = tid; h < p.Hkv; h += kSelThreads)
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
        const int32_t per = (n + kSelThreads - 1) / kSelThreads;
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
            const int32_t cnt = nret * ((Lb + p.P - 1) / p.P);
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
            for (int w = 0; w < kSelWarps; ++w) tot += scan[w];
            item_start[n] = tot;
        }
        __syncthreads();
    }
    const int32_t W = item_start[p.B];
    auto npages_of = [&](int32_t b) { return (item_len[b] + p.P - 1) / p.P; };
    auto seg_span = [&](int32_t s, int32_t& st, int32_t& len) {
        const int32_t b = s / p.Hkv, h = s - b * p.Hkv;
        const int32_t n = npages_of(b);
        const bool ret = p.head_kind[h] == DATTN_HEAD_RETRIEVAL;
        st = item_start[b] + ret_before[h] * n;
        len = ret ? n : 0;
    };
    auto locate = [&](int32_t t) {  // segment containing unit t
        int32_t lo = 0, hi = p.B - 1;
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (item_start[mid] <= t) lo = mid; else hi = mid - 1;
        }
        const int32_t n = npages_of(lo);
        const int32_t r = (t - item_start[lo]) / n;
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
            for (int r = tid; r < K; r += kSelThreads) p.selected[(int64_t)s * K + r] = -1;
    }
    if (t_begin >= t_end) return;

    const uint64_t pol = policy_evict_first();
    const int NT = kSelThreads;
    uint64_t* wbuf = reinterpret_cast<uint64_t*>(base + L.wbuf) + warp * L.wn;
    const int capw = L.wn - K;
    auto csync = [&]() { __syncthreads(); };
    auto wsync = [&]() { __syncwarp(); };
    auto warp_fold = [&](int cnt) {  // fold candidates wbuf[K .. K+cnt) into wbuf[0 .. K)
        for (int i = K + cnt + lane; i < L.wn; i += 32) wbuf[i] = 0ull;
        __syncwarp();
        bitonic_desc(wbuf, L.wn, lane, 32, wsync);
    };
    auto finalize = [&](int32_t seg) {  // sortbuf[0 .. K): top K keys -> ascending pages
        for (int i = tid; i < L.sn; i += NT)
            sortbuf[i] = i < K ? (sortbuf[i] & 0xFFFFFFFFull) * (sortbuf[i] != 0ull) : 0ull;
        csync();
        bitonic_desc(sortbuf, next_pow2(K), tid, NT, csync);  // low word desc = page asc
        for (int r = tid; r < K; r += NT) {
            const uint64_t kk = sortbuf[r];
            p.selected[(int64_t)seg * K + r] = kk ? (int32_t)(0xFFFFFFFFu - (uint32_t)kk) : -1;
        }
        csync();
    };

    // lane layout inside a warp group: row rr = lane / LPR, chunk c = lane % LPR
    const int c = lane % LPR, rr = lane / LPR;
    // rows of a unit: whole pages, at least one warp group
    const int unit_rows = LPG > RPW ? LPG : RPW;
    const int up = unit_rows / LPG;          // pages per unit
    const int ngu = unit_rows / RPW;         // warp groups per unit
    uint64_t qp2[HG][NPAIR], qn2[HG][NPAIR];  // the lane's query values: {ch 2i, ch 2i+1}

    int32_t a = t_begin;
    int32_t s = locate(t_begin);
    while (a < t_end) {
        int32_t sst, slen;
        seg_span(s, sst, slen);
        while (sst + slen <= a) { ++s; seg_span(s, sst, slen); }
        const int32_t pe = min(sst + slen, t_end);
        const int32_t b = s / p.Hkv, h = s - b * p.Hkv;
        const int32_t Lb = item_len[b];
        // the lane's query values, widened exactly, split by sign
#pragma unroll
        for (int j = 0; j < HG; ++j) {
            const bool okj = j < p.g;
            const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
                p.q + ((int64_t)b * p.Hq + h * p.g + (okj ? j : 0)) * D + c * CPL);
#pragma unroll
            for (int i = 0; i < NPAIR; ++i) {
                const uint32_t w = okj ? __ldg(qrow + i) : 0u;
                const float q0 = bf16_lo(w), q1 = bf16_hi(w);
                qp2[j][i] = pack_f32x2(q0 >= 0.f ? q0 : 0.f, q1 >= 0.f ? q1 : 0.f);
                qn2[j][i] = pack_f32x2(q0 >= 0.f ? 0.f : q0, q1 >= 0.f ? 0.f : q1);
            }
        }
        for (int i = lane; i < L.wn; i += 32) wbuf[i] = 0ull;
        __syncwarp();
        int cnt_c = 0;
        uint64_t thresh = 0ull;
        const int32_t* btrow = p.block_table + (int64_t)b * p.max_pages;
        // ---- blocks of pages: stage the block-table entries, then score ------------
        for (int32_t pb = a; pb < pe; pb += kSelBlockPages) {
            const int32_t nblk = min(kSelBlockPages, pe - pb);
            const int32_t pr0 = pb - sst;  // request-relative index of the block's first page
            for (int i = tid; i < nblk; i += NT) bt_blk[i] = __ldg(btrow + pr0 + i);
            csync();
            const int nunits = (nblk + up - 1) / up;
            const int ng = ((nunits - warp + kSelWarps - 1) / kSelWarps) * ngu;  // my groups
            // group k of this warp -> unit warp + 8*(k / ngu), part k % ngu
            auto row_of = [&](int k, int& pib, int& lp, bool& valid, int32_t& phys) {
                const int u = warp + kSelWarps * (k / ngu);
                const int r = u * unit_rows + (k % ngu) * RPW + rr;  // row in the block
                pib = r / LPG;
                lp = r - pib * LPG;
                valid = k < ng && pib < nblk && (pr0 + pib) * p.P + lp * 16 < Lb;
                phys = valid ? bt_blk[pib] : -1;
                if (valid && (phys < 0 || phys >= p.num_pages)) {
                    set_err(p.dev_err, phys < 0 ? DATTN_DEVERR_UNMAPPED_PAGE
                                                : DATTN_DEVERR_PAGE_OOB);
                    valid = false;
                }
            };
            auto issue = [&](int k, uint4 (&buf)[2 * NLD]) {
                int pib, lp;
                bool valid;
                int32_t phys;
                row_of(k, pib, lp, valid, phys);
                if (valid) {
                    const uint16_t* row = p.stats +
                        (((int64_t)phys * p.Hkv + h) * LPG + lp) * (2 * D) + c * CPL;
#pragma unroll
                    for (int i = 0; i < NLD; ++i) {
                        buf[i] = ldg_stream(row + i * 8, pol);
                        buf[NLD + i] = ldg_stream(row + D + i * 8, pol);
                    }
                }
            };
            float run = -__int_as_float(0x7f800000);  // running page max across a unit's groups
            auto process = [&](int k, const uint4 (&buf)[2 * NLD]) {
                if (k >= ng) return;  // warp-uniform
                int pib, lp;
                bool valid;
                int32_t phys;
                row_of(k, pib, lp, valid, phys);
                float best = -__int_as_float(0x7f800000);
                {
                    uint64_t acc[HG];
#pragma unroll
                    for (int j = 0; j < HG; ++j) acc[j] = 0ull;
                    const uint32_t* xw = reinterpret_cast<const uint32_t*>(&buf[0]);
                    const uint32_t* nw = reinterpret_cast<const uint32_t*>(&buf[NLD]);
#pragma unroll
                    for (int i = 0; i < NPAIR; ++i) {
                        const uint64_t kx2 = pack_f32x2(bf16_lo(xw[i]), bf16_hi(xw[i]));
                        const uint64_t kn2 = pack_f32x2(bf16_lo(nw[i]), bf16_hi(nw[i]));
#pragma unroll
                        for (int j = 0; j < HG; ++j) {
                            fma_f32x2(acc[j], qp2[j][i], kx2);
                            fma_f32x2(acc[j], qn2[j][i], kn2);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < HG; ++j) {
                        float ev, od;
                        unpack_f32x2(acc[j], ev, od);
                        float t = ev + od;
#pragma unroll
                        for (int off = 1; off < LPR; off <<= 1)
                            t = t + __shfl_xor_sync(0xffffffffu, t, off);
                        if (j < p.g) best = fmaxf(best, t);
                    }
                }
                if (!valid) best = -__int_as_float(0x7f800000);
                // page maximum over its logical pages (rows)
                if (LPG <= RPW) {
                    for (int off = LPR; off < LPR * LPG; off <<= 1)
                        best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, off));
                } else {
                    for (int off = LPR; off < 32; off <<= 1)
                        best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, off));
                    run = fmaxf(run, best);
                    best = run;
                    if ((k % ngu) != ngu - 1) return;  // the page continues in the next group
                    run = -__int_as_float(0x7f800000);
                }
                // one lane per page proposes the page's key
                const int u = warp + kSelWarps * (k / ngu);
                const int first_row = (k % ngu) * RPW + rr;  // row within the unit
                const int pib0 = (u * unit_rows + first_row) / LPG;
                const bool leader = c == 0 && (first_row % LPG == 0 || LPG > RPW) &&
                                    (LPG <= RPW || rr == 0) && pib0 < nblk;
                uint64_t key = 0ull;
                if (leader && best != -__int_as_float(0x7f800000)) key = make_key(best, pr0 + pib0);
                const bool take = key > thresh;
                const uint32_t bal = __ballot_sync(0xffffffffu, take);
                if (take) wbuf[K + cnt_c + __popc(bal & ((1u << lane) - 1u))] = key;
                cnt_c += __popc(bal);
                __syncwarp();
                if (cnt_c > capw - 32) {
                    warp_fold(cnt_c);
                    cnt_c = 0;
                    thresh = wbuf[K - 1];
                }
            };
            // three groups in flight per warp
            uint4 b0[2 * NLD], b1[2 * NLD], b2[2 * NLD];
            issue(0, b0);
            issue(1, b1);
            issue(2, b2);
            for (int k = 0; k < ng; k += 3) {
                process(k, b0);
                issue(k + 3, b0);
                process(k + 1, b1);
                issue(k + 4, b1);
                process(k + 2, b2);
                issue(k + 5, b2);
            }
            csync();  // bt_blk is rewritten by the next block
        }
        if (cnt_c > 0) warp_fold(cnt_c);
        csync();
        // merge the warps' lists of this piece
        for (int i = tid; i < L.sn; i += NT) {
            const int w = i / K, r = i - w * K;
            sortbuf[i] = w < kSelWarps ? reinterpret_cast<uint64_t*>(base + L.wbuf)[w * L.wn + r]
                                       : 0ull;
        }
        csync();
        bitonic_desc(sortbuf, L.sn, tid, NT, csync);
        const bool whole = (a == sst) && (pe == sst + slen);
        if (whole) {
            finalize(s);
        } else {
            uint64_t* my = p.slots + (int64_t)(cta + s) * K;
            for (int r = tid; r < K; r += NT) my[r] = sortbuf[r];
            csync();
            const int32_t c_first = split_owner(sst, W, Gw);
            const int32_t c_last = split_owner(sst + slen - 1, W, Gw);
            const int32_t npieces = c_last - c_first + 1;
            if (tid == 0) {
                __threadfence();
                const int32_t prev = atomicAdd(p.counters + s, 1);
                *last_flag = (prev == npieces - 1) ? 1 : 0;
                if (prev == npieces - 1) p.counters[s] = 0;
            }
            csync();
            if (*last_flag) {
                __threadfence();
                // fold the pieces in groups: sortbuf = [top K | up to (sn - K) new keys]
                for (int i = tid; i < L.sn; i += NT) sortbuf[i] = 0ull;
                csync();
                const int per_fold = (L.sn - K) / K;
                for (int32_t q0 = 0; q0 < npieces; q0 += per_fold) {
                    const int32_t nq = min(per_fold, npieces - q0);
                    for (int i = tid; i < L.sn - K; i += NT) {
                        const int32_t qq = q0 + i / K, r = i % K;
                        sortbuf[K + i] = (i < nq * K)
                            ? __ldcg(reinterpret_cast<const unsigned long long*>(
                                  p.slots + (int64_t)(c_first + qq + s) * K + r))
                            : 0ull;
                    }
                    csync();
                    bitonic_desc(sortbuf, L.sn, tid, NT, csync);
                }
                finalize(s);
            }
        }
        csync();
        a = pe;
    }
}

template <int D, int CPL, int HG>
int sel_prepare(uint32_t smem) {
    static int max_set = 0;
    if ((int)smem > max_set) {
        if (cudaFuncSetAttribute(page_select_kernel<D, CPL, HG>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return -1;
        max_set = (int)smem;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, page_select_kernel<D, CPL, HG>,
                                                      kSelThreads, smem) != cudaSuccess)
        return 1;
    return n < 1 ? 1 : n;
}

template <int D, int CPL, int HG>
cudaError_t sel_launch(int32_t G, uint32_t smem, cudaStream_t stream, const SelParams& p) {
    return launch_pdl(page_select_kernel<D, CPL, HG>, dim3(G), dim3(kSelThreads), smem, stream,
                      p);
}

}  // namespace

size_t select_workspace_bytes(int32_t nseg, int32_t top_k, int32_t G) {
    const size_t counters = ((size_t)nseg * 4 + 255) & ~(size_t)255;
    return counters + (size_t)(G + nseg) * top_k * 8;
}

dattn_status_t launch_page_select(const dattn_kv_layout& Lay, const uint16_t* stats,
                                  const uint16_t* q, int32_t B, int32_t Hq,
                                  const int32_t* seq_lens, const int8_t* head_kind,
                                  int32_t top_k, int32_t* selected, void* ws, size_t ws_bytes,
                                  int32_t num_splits, int32_t* dev_err, cudaStream_t stream,
                                  int64_t units_bound) {
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
    p.nseg = B * p.Hkv;
    p.dev_err = dev_err;
    const int D = Lay.head_dim;
    const bool wide = p.g > 4;  // 8 channels x 8 heads per lane instead of 16 x 4
    const SelSmem L = sel_smem_layout(B, p.Hkv, top_k);
    if (L.total > 227u * 1024u) return DATTN_ERR_UNSUPPORTED;
    int occ;
    if (D == 64) occ = wide ? sel_prepare<64, 8, 8>(L.total) : sel_prepare<64, 16, 4>(L.total);
    else occ = wide ? sel_prepare<128, 8, 8>(L.total) : sel_prepare<128, 16, 4>(L.total);
    if (occ < 0) return DATTN_ERR_CUDA;
    const int32_t G = choose_splits(units_bound * 4, num_splits, occ);
    const size_t counters = ((size_t)p.nseg * 4 + 255) & ~(size_t)255;
    if (ws == nullptr || ws_bytes < select_workspace_bytes(p.nseg, top_k, G) ||
        (reinterpret_cast<uintptr_t>(ws) & 255))
        return DATTN_ERR_WORKSPACE;
    p.counters = static_cast<int32_t*>(ws);
    p.slots = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(ws) + counters);
    cudaError_t e;
    if (D == 64)
        e = wide ? sel_launch<64, 8, 8>(G, L.total, stream, p)
                 : sel_launch<64, 16, 4>(G, L.total, stream, p);
    else
        e = wide ? sel_launch<128, 8, 8>(G, L.total, stream, p)
                 : sel_launch<128, 16, 4>(G, L.total, stream, p);
    return e == cudaSuccess ? DATTN_OK : DATTN_ERR_CUDA;
}

}  // namespace dattn
