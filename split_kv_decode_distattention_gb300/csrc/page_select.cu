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
// GB300 design. The statistics scan is HBM-bound: every 16 decode steps it reads all k_max
// and k_min of the retrieval heads. The physical pages of all retrieval (request, KV head)
// pairs are laid end to end and cut into equal contiguous ranges, one per CTA. A producer
// warp bulk-copies each page's statistics tile (contiguous in HBM) into a stage padded by 16
// bytes per page, so the eight lanes of a shared-memory phase, which read eight different
// pages, hit eight different banks. Four consumer warps score a stage together, keep the
// pages that beat the running K-th key in a candidate buffer, and fold candidates into the
// top K with a 512-entry bitonic sort in shared memory. A head split across CTAs leaves
// each CTA's top K in the workspace, and the CTA that arrives last merges them.
#include "common.cuh"
#include "internal.h"

namespace dattn {

namespace {

constexpr int kSelStages = 4;
constexpr int kSortN = 512;
constexpr int kSelThreads = kAttnThreads;  // 4 consumer warps + 1 producer warp

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
    int32_t npg;          // physical pages per stage (power of two, <= 32)
    uint32_t page_bytes;  // statistics bytes of one (page, head): (P/16) * 2 * D * 2
    int32_t* dev_err;
};

struct SelSmem {
    uint32_t stage_bytes, stages, bars, meta, flags, qs, scr, sortbuf, ret_before, ret_heads,
        item_start, item_len, scan, total;
};

__host__ __device__ inline SelSmem sel_smem_layout(int D, int g, int P, int npg, int B, int Hkv) {
    SelSmem s;
    const uint32_t page_bytes = (uint32_t)(P / 16) * 2u * D * 2u;
    s.stage_bytes = (uint32_t)npg * (page_bytes + 16u);
    uint32_t o = 0;
    s.stages = o;     o += kSelStages * s.stage_bytes;
    s.bars = o;       o += 2u * kSelStages * 8u;
    s.meta = o;       o += kSelStages * 4u;
    s.flags = o;      o += 16u;
    s.qs = o;         o += (uint32_t)(g * D) * 4u;
    s.scr = o;        o += (uint32_t)(npg * (P / 16) * g) * 4u;
    o = (o + 15u) & ~15u;
    s.sortbuf = o;    o += kSortN * 8u;
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

// Bitonic sort of buf[0..n) into descending order by the 128 consumer threads (n a power of
// two). Ends with a barrier.
__device__ void bitonic_desc(uint64_t* buf, int n, int ctid) {
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int idx = ctid; idx < (n >> 1); idx += kConsumerWarps * 32) {
                const int i = 2 * j * (idx / j) + (idx % j);
                const int l = i + j;
                const uint64_t x = buf[i], y = buf[l];
                const bool desc = (i & k) == 0;
                if (desc ? (x < y) : (x > y)) {
                    buf[i] = y;
                    buf[l] = x;
                }
            }
            named_bar_sync(1, kConsumerWarps * 32);
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kSelThreads) page_select_kernel(const __grid_constant__ SelParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_off = smem_u32(smem_raw);
    uint8_t* base = smem_raw + (((raw_off + 127u) & ~127u) - raw_off);
    const SelSmem L = sel_smem_layout(D, p.g, p.P, p.npg, p.B, p.Hkv);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int32_t G = gridDim.x, cta = blockIdx.x;
    const int LPG = p.P >> 4;
    const uint32_t bars = smem_u32(base + L.bars);
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto empty_bar = [&](int s) { return bars + 8u * (kSelStages + s); };
    uint32_t* meta = reinterpret_cast<uint32_t*>(base + L.meta);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base + L.flags);
    int* cand_count = reinterpret_cast<int*>(base + L.flags + 4);
    int* last_flag = reinterpret_cast<int*>(base + L.flags + 8);
    float* qs = reinterpret_cast<float*>(base + L.qs);
    float* scr = reinterpret_cast<float*>(base + L.scr);
    uint64_t* sortbuf = reinterpret_cast<uint64_t*>(base + L.sortbuf);
    int32_t* ret_before = reinterpret_cast<int32_t*>(base + L.ret_before);
    int32_t* ret_heads = reinterpret_cast<int32_t*>(base + L.ret_heads);
    int32_t* item_start = reinterpret_cast<int32_t*>(base + L.item_start);
    int32_t* item_len = reinterpret_cast<int32_t*>(base + L.item_len);
    int32_t* scan = reinterpret_cast<int32_t*>(base + L.scan);

    // ---------------------------------------------------------------- setup
    if (tid == 0) {
        for (int s = 0; s < kSelStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
        int32_t r = 0;
        for (int h = 0; h < p.Hkv; ++h) {
            ret_before[h] = r;
            if (p.head_kind[h] == DATTN_HEAD_RETRIEVAL) ret_heads[r++] = h;
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
            for (int w = 0; w < kSelThreads / 32; ++w) tot += scan[w];
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
            for (int r = tid; r < p.top_k; r += kSelThreads) p.selected[(int64_t)s * p.top_k + r] = -1;
    }
    if (t_begin >= t_end) return;

    const uint32_t stage0 = smem_u32(base + L.stages);
    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer warp
        const uint64_t pol = policy_evict_first();
        int32_t u = 0;  // stage uses so far
        int32_t a = t_begin;
        int32_t s = locate(t_begin);
        bool stop = false;
        while (a < t_end && !stop) {
            int32_t sst, slen;
            seg_span(s, sst, slen);
            while (sst + slen <= a) { ++s; seg_span(s, sst, slen); }
            const int32_t pe = min(sst + slen, t_end);
            const int32_t b = s / p.Hkv, h = s - b * p.Hkv;
            for (int32_t x = a; x < pe && !stop; x += p.npg, ++u) {
                const int stg = u % kSelStages;
                bool ok = true;
                if (lane == 0 && u >= kSelStages)
                    ok = mbar_wait(empty_bar(stg), ((u / kSelStages) - 1) & 1, abort_flag, p.dev_err);
                stop = __shfl_sync(0xffffffffu, ok ? 0 : 1, 0) != 0;
                if (stop) break;
                const int32_t cnt = min(p.npg, pe - x);
                bool valid = false;
                int32_t page = 0;
                if (lane < cnt) {
                    const int32_t pi = x - sst + lane;  // request-relative page index
                    page = p.block_table[(int64_t)b * p.max_pages + pi];
                    if (page < 0) set_err(p.dev_err, DATTN_DEVERR_UNMAPPED_PAGE);
                    else if (page >= p.num_pages) set_err(p.dev_err, DATTN_DEVERR_PAGE_OOB);
                    else valid = true;
                }
                const uint32_t mask = __ballot_sync(0xffffffffu, valid);
                if (lane == 0) {
                    meta[stg] = mask;
                    if (mask) mbar_arrive_expect_tx(full_bar(stg), __popc(mask) * p.page_bytes);
                    else mbar_arrive(full_bar(stg));
                }
                __syncwarp();
                if (valid) {
                    const uint16_t* src = p.stats + ((int64_t)page * p.Hkv + h) * (p.page_bytes / 2);
                    bulk_load(stage0 + stg * L.stage_bytes + lane * (p.page_bytes + 16u), src,
                              p.page_bytes, full_bar(stg), pol);
                }
            }
            a = pe;
        }
        if (lane == 0 && *abort_flag) {  // bounded wait for copies still in flight
            for (int32_t k = max(0, u - kSelStages); k < u; ++k) {
                const unsigned long long t0 = global_timer_ns();
                while (!mbar_try_wait(full_bar(k % kSelStages), (k / kSelStages) & 1) &&
                       global_timer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumer warps
    const int ctid = tid;
    const int K = p.top_k;
    const int nitem = p.npg * LPG * p.g;
    int32_t u = 0;
    int32_t a = t_begin;
    int32_t s = locate(t_begin);
    auto fold = [&]() {  // fold the candidates into the running top K
        const int c = *cand_count;
        for (int i = K + c + ctid; i < kSortN; i += kConsumerWarps * 32) sortbuf[i] = 0ull;
        named_bar_sync(1, kConsumerWarps * 32);
        bitonic_desc(sortbuf, kSortN, ctid);
        if (ctid == 0) *cand_count = 0;
        named_bar_sync(1, kConsumerWarps * 32);
    };
    auto finalize = [&](int32_t seg) {  // sortbuf[0..K) holds the top K keys
        for (int i = ctid; i < kSortN; i += kConsumerWarps * 32)
            sortbuf[i] = i < K ? (sortbuf[i] & 0xFFFFFFFFull) * (sortbuf[i] != 0ull) : 0ull;
        named_bar_sync(1, kConsumerWarps * 32);
        int n2 = 1;
        while (n2 < K) n2 <<= 1;
        bitonic_desc(sortbuf, n2, ctid);  // descending low word = ascending page index
        for (int r = ctid; r < K; r += kConsumerWarps * 32) {
            const uint64_t kk = sortbuf[r];
            p.selected[(int64_t)seg * K + r] = kk ? (int32_t)(0xFFFFFFFFu - (uint32_t)kk) : -1;
        }
        named_bar_sync(1, kConsumerWarps * 32);
    };

    while (a < t_end) {
        int32_t sst, slen;
        seg_span(s, sst, slen);
        while (sst + slen <= a) { ++s; seg_span(s, sst, slen); }
        const int32_t pe = min(sst + slen, t_end);
        const int32_t b = s / p.Hkv, h = s - b * p.Hkv;
        const int32_t Lb = item_len[b];
        // queries of the group, widened exactly to fp32
        for (int i = ctid; i < p.g * D; i += kConsumerWarps * 32) {
            const int j = i / D, d = i - j * D;
            qs[i] = __uint_as_float((uint32_t)p.q[((int64_t)b * p.Hq + h * p.g + j) * D + d] << 16);
        }
        for (int i = ctid; i < kSortN; i += kConsumerWarps * 32) sortbuf[i] = 0ull;
        if (ctid == 0) *cand_count = 0;
        named_bar_sync(1, kConsumerWarps * 32);
        uint64_t thresh = 0ull;
        for (int32_t x = a; x < pe; x += p.npg, ++u) {
            const int stg = u % kSelStages;
            const bool ok = mbar_wait(full_bar(stg), (u / kSelStages) & 1, abort_flag, p.dev_err);
            const uint32_t mask = ok ? meta[stg] : 0u;
            const int32_t cnt = min(p.npg, pe - x);
            const uint8_t* sb = base + L.stages + stg * L.stage_bytes;
            // items (page-fastest): it = (lp * g + j) * npg + i
            for (int it0 = ctid; it0 < nitem; it0 += 2 * kConsumerWarps * 32) {
                float acc[2] = {0.f, 0.f};
                const float* qrow[2];
                const uint8_t* row[2];
                bool val[2];
                int idx[2];
#pragma unroll
                for (int w = 0; w < 2; ++w) {
                    const int it = it0 + w * kConsumerWarps * 32;
                    idx[w] = it;
                    const int i = it % p.npg, r = it / p.npg;
                    const int lp = r / p.g, j = r - lp * p.g;
                    const int32_t pi = x - sst + i;
                    val[w] = it < nitem && i < cnt && ((mask >> i) & 1u) &&
                             (pi * p.P + lp * 16 < Lb);
                    row[w] = sb + i * (p.page_bytes + 16u) + lp * (2 * D * 2);
                    qrow[w] = qs + j * D;
                }
                if (val[0] || val[1]) {
#pragma unroll 2
                    for (int d8 = 0; d8 < D / 8; ++d8) {
#pragma unroll
                        for (int w = 0; w < 2; ++w) {
                            if (!val[w]) continue;
                            const uint4 mx = *reinterpret_cast<const uint4*>(row[w] + d8 * 16);
                            const uint4 mn = *reinterpret_cast<const uint4*>(row[w] + D * 2 + d8 * 16);
                            const uint32_t xs[4] = {mx.x, mx.y, mx.z, mx.w};
                            const uint32_t ns[4] = {mn.x, mn.y, mn.z, mn.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const float q0 = qrow[w][d8 * 8 + 2 * e];
                                const float q1 = qrow[w][d8 * 8 + 2 * e + 1];
                                acc[w] = fmaf(q0, q0 >= 0.f ? bf16_lo(xs[e]) : bf16_lo(ns[e]), acc[w]);
                                acc[w] = fmaf(q1, q1 >= 0.f ? bf16_hi(xs[e]) : bf16_hi(ns[e]), acc[w]);
                            }
                        }
                    }
                }
#pragma unroll
                for (int w = 0; w < 2; ++w)
                    if (idx[w] < nitem) scr[idx[w]] = val[w] ? acc[w] : -__int_as_float(0x7f800000);
            }
            named_bar_sync(1, kConsumerWarps * 32);
            if (ctid == 0) mbar_arrive(empty_bar(stg));  // the stage has been read
            // physical-page keys; keep those above the running K-th key
            for (int i = ctid; i < cnt; i += kConsumerWarps * 32) {
                float best = -__int_as_float(0x7f800000);
                bool any = false;
                for (int r = 0; r < LPG * p.g; ++r) {
                    const int it = r * p.npg + i;
                    const int lp = r / p.g;
                    if ((x - sst + i) * p.P + lp * 16 < Lb && ((mask >> i) & 1u)) {
                        best = any ? fmaxf(best, scr[it]) : scr[it];
                        any = true;
                    }
                }
                if (any) {
                    const uint64_t key = make_key(best, x - sst + i);
                    if (key > thresh) {
                        const int slot = atomicAdd(cand_count, 1);
                        sortbuf[K + slot] = key;
                    }
                }
            }
            named_bar_sync(1, kConsumerWarps * 32);
            if (*cand_count > kSortN - K - p.npg) {
                fold();
                thresh = sortbuf[K - 1];
            }
        }
        if (*cand_count > 0) fold();
        const bool whole = (a == sst) && (pe == sst + slen);
        if (whole) {
            finalize(s);
        } else {
            uint64_t* my = p.slots + (int64_t)(cta + s) * K;
            for (int r = ctid; r < K; r += kConsumerWarps * 32) my[r] = sortbuf[r];
            named_bar_sync(1, kConsumerWarps * 32);
            const int32_t c_first = split_owner(sst, W, Gw);
            const int32_t c_last = split_owner(sst + slen - 1, W, Gw);
            const int32_t npieces = c_last - c_first + 1;
            if (ctid == 0) {
                __threadfence();
                const int32_t prev = atomicAdd(p.counters + s, 1);
                *last_flag = (prev == npieces - 1) ? 1 : 0;
                if (prev == npieces - 1) p.counters[s] = 0;
            }
            named_bar_sync(1, kConsumerWarps * 32);
            if (*last_flag) {
                __threadfence();
                for (int i = ctid; i < kSortN; i += kConsumerWarps * 32) sortbuf[i] = 0ull;
                named_bar_sync(1, kConsumerWarps * 32);
                const int per_fold = (kSortN - K) / K;
                for (int32_t q0 = 0; q0 < npieces; q0 += per_fold) {
                    const int32_t nq = min(per_fold, npieces - q0);
                    for (int i = ctid; i < nq * K; i += kConsumerWarps * 32) {
                        const int32_t qq = q0 + i / K, r = i % K;
                        sortbuf[K + i] = __ldcg(reinterpret_cast<const unsigned long long*>(
                            p.slots + (int64_t)(c_first + qq + s) * K + r));
                    }
                    if (ctid == 0) *cand_count = nq * K;
                    named_bar_sync(1, kConsumerWarps * 32);
                    fold();
                }
                finalize(s);
            }
        }
        named_bar_sync(1, kConsumerWarps * 32);
        a = pe;
    }
}

int pick_npg(uint32_t page_bytes) {
    int n = 32;
    while (n > 1 && (uint32_t)n * (page_bytes + 16u) > 34000u) n >>= 1;
    return n;
}

template <int D>
int sel_occupancy(uint32_t smem) {
    static int max_set = 0;
    if ((int)smem > max_set) {
        if (cudaFuncSetAttribute(page_select_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return -1;
        max_set = (int)smem;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, page_select_kernel<D>, kSelThreads,
                                                      smem) != cudaSuccess)
        return 1;
    return n < 1 ? 1 : n;
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
    const int D = Lay.head_dim;
    p.page_bytes = (uint32_t)(p.P / 16) * 2u * D * 2u;
    p.npg = pick_npg(p.page_bytes);
    p.dev_err = dev_err;
    const SelSmem L = sel_smem_layout(D, p.g, p.P, p.npg, B, p.Hkv);
    const int occ = D == 64 ? sel_occupancy<64>(L.total) : sel_occupancy<128>(L.total);
    if (occ < 0) return DATTN_ERR_CUDA;
    const int32_t G = choose_splits(units_bound * 4, num_splits, occ);
    const size_t counters = ((size_t)p.nseg * 4 + 255) & ~(size_t)255;
    if (ws == nullptr || ws_bytes < select_workspace_bytes(p.nseg, top_k, G) ||
        (reinterpret_cast<uintptr_t>(ws) & 255))
        return DATTN_ERR_WORKSPACE;
    p.counters = static_cast<int32_t*>(ws);
    p.slots = reinterpret_cast<uint64_t*>(static_cast<uint8_t*>(ws) + counters);
    if (D == 64)
        page_select_kernel<64><<<G, kSelThreads, L.total, stream>>>(p);
    else
        page_select_kernel<128><<<G, kSelThreads, L.total, stream>>>(p);
    return cudaGetLastError() == cudaSuccess ? DATTN_OK : DATTN_ERR_CUDA;
}

}  // namespace dattn
