// Paged KV append with logical-page statistics (dattn_kv_append).
//
// "LoongServe: Efficiently Serving Long-Context Large Language Models with Elastic Sequence
// Parallelism", §4.2: in distributed decoding the master saves the new token's KV in its
// local KV pool. "LLM长序列服务优化：LServe的块稀疏注意力技术", §3.1.2: the per-channel
// k_max / k_min of each 16-token logical page are computed when the KV cache is written,
// so decoding pays nothing for them.
//
// Each CTA owns a window of 64 token positions aligned to logical pages (16 tokens). It
// copies the K and V rows of its tokens with 16-byte vectors into their (page, head, slot)
// places, then folds its tokens into the statistics of the logical pages it covers.
// Because the windows are aligned to logical pages, no two CTAs touch the same logical page,
// so the statistics need no atomics and come out the same on every run.
#include "common.cuh"
#include "internal.h"

namespace dattn {

namespace {

constexpr int kAppendThreads = 128;
constexpr int kAppendWindow = 64;  // token positions per CTA, a multiple of 16

__device__ __forceinline__ float bf(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

template <int D>
__global__ void __launch_bounds__(kAppendThreads)
kv_append_kernel(dattn_kv_layout L, uint16_t* __restrict__ k_pool, uint16_t* __restrict__ v_pool,
                 uint16_t* __restrict__ stats, const uint16_t* __restrict__ k_new,
                 const uint16_t* __restrict__ v_new, int32_t T, int32_t* seq_lens,
                 int32_t update_in_place, int32_t* dev_err) {
    const int32_t b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
    const int32_t Hkv = L.num_kv_heads, P = L.page_size;
    grid_dependency_wait();  // the previous kernel may still read the pool or the lengths
    grid_launch_dependents();
    const int32_t pos0 = seq_lens[b];
    if (pos0 < 0) {
        if (tid == 0) set_err(dev_err, DATTN_DEVERR_LEN_OOB);
        return;
    }
    const int32_t base = pos0 - (pos0 & 15);
    const int32_t p_lo = max(pos0, base + c * kAppendWindow);
    const int32_t p_hi = min(pos0 + T, base + (c + 1) * kAppendWindow);
    const int32_t* bt = L.block_table + (int64_t)b * L.max_pages_per_req;

    if (p_lo < p_hi) {
        // ---- K and V rows: 16-byte vectors ---------------------------------------------
        constexpr int VPR = D / 8;  // vectors per (token, head) row
        const int32_t nvec = (p_hi - p_lo) * Hkv * VPR;
        for (int32_t v = tid; v < nvec; v += kAppendThreads) {
            const int32_t t = p_lo + v / (Hkv * VPR);
            const int32_t rem = v - (t - p_lo) * (Hkv * VPR);
            const int32_t h = rem / VPR, dv = rem - h * VPR;
            const int32_t lp = t / P;
            if (lp >= L.max_pages_per_req) {
                set_err(dev_err, DATTN_DEVERR_LEN_OOB);
                continue;
            }
            const int32_t page = bt[lp];
            if (page < 0) {
                set_err(dev_err, DATTN_DEVERR_UNMAPPED_PAGE);
                continue;
            }
            if (page >= L.num_pages) {
                set_err(dev_err, DATTN_DEVERR_PAGE_OOB);
                continue;
            }
            const int64_t src = (((int64_t)b * T + (t - pos0)) * Hkv + h) * D + dv * 8;
            const int64_t dst = (((int64_t)page * Hkv + h) * P + (t - lp * P)) * D + dv * 8;
            *reinterpret_cast<uint4*>(k_pool + dst) = *reinterpret_cast<const uint4*>(k_new + src);
            *reinterpret_cast<uint4*>(v_pool + dst) = *reinterpret_cast<const uint4*>(v_new + src);
        }
        // ---- statistics of the logical pages in this window ------------------------------
        if (stats != nullptr) {
            const int32_t lq0 = p_lo >> 4, lq1 = (p_hi - 1) >> 4;
            constexpr int PAIRS = D / 2;
            const int32_t nwork = (lq1 - lq0 + 1) * Hkv * PAIRS;
            for (int32_t w = tid; w < nwork; w += kAppendThreads) {
                const int32_t lq = lq0 + w / (Hkv * PAIRS);
                const int32_t rem = w - (lq - lq0) * (Hkv * PAIRS);
                const int32_t h = rem / PAIRS, dp = rem - h * PAIRS;
                const int32_t first = lq * 16;
                const int32_t ta = max(first, p_lo), tb = min(first + 16, p_hi);
                const int32_t lp = first / P;
                if (lp >= L.max_pages_per_req) continue;  // flagged by the copy above
                const int32_t page = bt[lp];
                if (page < 0 || page >= L.num_pages) continue;
                uint16_t* st = stats + ((((int64_t)page * Hkv + h) * (P / 16) +
                                         (first - lp * P) / 16) * 2) * D + 2 * dp;
                const uint16_t* kr = k_new + (((int64_t)b * T + (ta - pos0)) * Hkv + h) * D + 2 * dp;
                const int64_t tstride = (int64_t)Hkv * D;
                uint16_t mx0, mx1, mn0, mn1;
                int32_t t = ta;
                if (ta == first) {  // this append opens the logical page
                    const uint32_t k2 = *reinterpret_cast<const uint32_t*>(kr);
                    mx0 = mn0 = (uint16_t)(k2 & 0xffff);
                    mx1 = mn1 = (uint16_t)(k2 >> 16);
                    ++t;
                } else {
                    const uint32_t x2 = *reinterpret_cast<const uint32_t*>(st);
                    const uint32_t n2 = *reinterpret_cast<const uint32_t*>(st + D);
                    mx0 = (uint16_t)(x2 & 0xffff); mx1 = (uint16_t)(x2 >> 16);
                    mn0 = (uint16_t)(n2 & 0xffff); mn1 = (uint16_t)(n2 >> 16);
                }
                for (; t < tb; ++t) {
                    const uint32_t k2 =
                        *reinterpret_cast<const uint32_t*>(kr + (int64_t)(t - ta) * tstride);
                    const uint16_t a = (uint16_t)(k2 & 0xffff), z = (uint16_t)(k2 >> 16);
                    // strict comparisons: on a tie the earlier value stays
                    if (bf(a) > bf(mx0)) mx0 = a;
                    if (bf(a) < bf(mn0)) mn0 = a;
                    if (bf(z) > bf(mx1)) mx1 = z;
                    if (bf(z) < bf(mn1)) mn1 = z;
                }
                *reinterpret_cast<uint32_t*>(st) = (uint32_t)mx0 | ((uint32_t)mx1 << 16);
                *reinterpret_cast<uint32_t*>(st + D) = (uint32_t)mn0 | ((uint32_t)mn1 << 16);
            }
        }
    }
    if (update_in_place) {
        __syncthreads();  // every thread has read seq_lens[b]
        if (tid == 0) seq_lens[b] = pos0 + T;
    }
}

__global__ void advance_lengths_kernel(int32_t* seq_lens, int32_t B, int32_t T) {
    grid_dependency_wait();
    grid_launch_dependents();
    const int32_t b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B && seq_lens[b] >= 0) seq_lens[b] += T;
}

}  // namespace

dattn_status_t launch_kv_append(const dattn_kv_layout& L, uint16_t* k_pool, uint16_t* v_pool,
                                uint16_t* stats, const uint16_t* k_new, const uint16_t* v_new,
                                int32_t B, int32_t T, int32_t* seq_lens, int32_t* dev_err,
                                cudaStream_t stream) {
    if (B == 0 || T == 0) return DATTN_OK;
    // a window of 64 aligned positions holds all T tokens whatever seq_lens % 16 is
    const bool single = T + 15 <= kAppendWindow;
    const int32_t nwin = single ? 1 : (T + 15 + kAppendWindow - 1) / kAppendWindow;
    const dim3 grid(nwin, B);
    const int32_t inplace = single ? 1 : 0;
    cudaError_t e;
    if (L.head_dim == 64)
        e = launch_pdl(kv_append_kernel<64>, grid, dim3(kAppendThreads), 0, stream, L, k_pool,
                       v_pool, stats, k_new, v_new, T, seq_lens, inplace, dev_err);
    else
        e = launch_pdl(kv_append_kernel<128>, grid, dim3(kAppendThreads), 0, stream, L, k_pool,
                       v_pool, stats, k_new, v_new, T, seq_lens, inplace, dev_err);
    if (e != cudaSuccess) return DATTN_ERR_CUDA;
    if (!single) {
        if (launch_pdl(advance_lengths_kernel, dim3((B + 255) / 256), dim3(256), 0, stream,
                       seq_lens, B, T) != cudaSuccess)
            return DATTN_ERR_CUDA;
    }
    return DATTN_OK;
}

}  // namespace dattn
