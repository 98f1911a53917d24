// Paged KV append with logical-page statistics (dattn_kv_append).
//
// "LoongServe: Efficiently Serving Long-Context Large Language Models with Elastic Sequence
// Parallelism", §4.2: in distributed decoding the master saves the new token's KV in its
// local KV pool. "LLM长序列服务优化：LServe的块稀疏注意力技术", §3.1.2: the per-channel
// k_max / k_min of each 16-token logical page are computed when the KV cache is written,
// so decoding pays nothing for them.
//
// Each CTA owns a window of 64 token positions aligned to logical pages (16 tokens), and
// each thread one (KV head, 8-channel chunk) of every token in it: it copies that chunk of
// the K and V rows with 16-byte vectors into their (page, head, slot) places and folds the
// same K chunk into the statistics of the logical page, keeping the running k_max / k_min
// of the open logical page in registers. Because the windows are aligned to logical
// pages, no two CTAs touch the same logical page, so the statistics need no atomics and
// come out the same on every run.
//
// The 8-bit pool (FP8 E4M3 codes, one fp32 scale per (token, KV head) row; the retrieval
// cache of "LLM长序列服务优化：LServe的块稀疏注意力技术" §3.2.1 is quantized at 2-8 bits):
// the d/8 threads of one row sit in consecutive lanes, so the row's max |x| is a shuffle
// reduction among them. scale = max|x| / 448 and each code is E4M3(x / scale), both
// divisions in IEEE fp32, the conversion rounding to nearest even with saturation. The
// statistics are still taken from the bf16 key.
//
// The 4-bit pool (the streaming-head cache of that section is 4-bit): scale = max|x| / 7 and
// each code is x / scale rounded to the nearest integer (ties to even) in [-7, 7], both
// divisions in IEEE fp32, stored as the nibble code + 8 with channel 2j in the low nibble of
// byte j. A thread's 8 channels become one 32-bit word.
//
// The mixed pool quantizes each KV head's rows in that head's format (8-bit or 4-bit) and
// writes them to the region of that format, at the head's index among its format's heads.
#include "common.cuh"
#include "internal.h"

namespace dattn {

namespace {

constexpr int kAppendMaxThreads = 512;  // one thread per (KV head, 8-channel chunk)
constexpr int kAppendWindow = 64;  // token positions per CTA, a multiple of 16

template <int D, int FMT>
__global__ void __launch_bounds__(kAppendMaxThreads)
kv_append_kernel(dattn_kv_layout L, const __grid_constant__ KvHeadFormats hf,
                 void* __restrict__ k_pool_v, void* __restrict__ v_pool_v,
                 uint16_t* __restrict__ stats, const uint16_t* __restrict__ k_new,
                 const uint16_t* __restrict__ v_new, int32_t T, int32_t* seq_lens,
                 int32_t update_in_place, int32_t* dev_err) {
    constexpr int VPR = D / 8;  // 8-channel chunks per (token, head) row
    const int32_t b = blockIdx.y, c = blockIdx.x, tid = threadIdx.x;
    const int32_t Hkv = L.num_kv_heads, P = L.page_size;
    if (tid == 0) prefetch_l2_range(seq_lens + b, 4u, 0, 1);  // the length is read first
    grid_dependency_wait();  // the previous kernel may still read the pool or the lengths
    grid_launch_dependents();
    // In a single-window launch the CTA takes the new tokens 0 .. T-1 whatever seq_lens
    // holds, so the first token's K/V chunk is loaded while the length is still in flight.
    const bool single = update_in_place != 0;
    const int64_t tstride = (int64_t)Hkv * D;  // elements between consecutive new tokens
    const uint16_t* kb = k_new + (int64_t)b * T * tstride;
    const uint16_t* vb = v_new + (int64_t)b * T * tstride;
    uint4 k0 = make_uint4(0u, 0u, 0u, 0u), v0 = k0;
    if (single && tid < Hkv * VPR) {
        k0 = *reinterpret_cast<const uint4*>(kb + (int64_t)tid * 8);
        v0 = *reinterpret_cast<const uint4*>(vb + (int64_t)tid * 8);
    }
    const int32_t pos0 = seq_lens[b];
    if (pos0 < 0) {
        if (tid == 0) set_err(dev_err, DATTN_DEVERR_LEN_OOB);
        return;
    }
    const int32_t base = pos0 - (pos0 & 15);
    const int32_t i_lo = max(pos0, base + c * kAppendWindow) - pos0;  // new-token range
    const int32_t i_hi = min(pos0 + T, base + (c + 1) * kAppendWindow) - pos0;
    const int32_t* bt = L.block_table + (int64_t)b * L.max_pages_per_req;
    const int32_t lpg = P >> 4;
    uint16_t* k_pool = static_cast<uint16_t*>(k_pool_v);
    uint16_t* v_pool = static_cast<uint16_t*>(v_pool_v);
    uint8_t* k_code = static_cast<uint8_t*>(k_pool_v);
    uint8_t* v_code = static_cast<uint8_t*>(v_pool_v);

    for (int32_t item = tid; item < Hkv * VPR && i_lo < i_hi; item += blockDim.x) {
        // lanes of this warp inside the loop: a prefix of the warp, whole rows only
        const int32_t warp_items = Hkv * VPR - (item - (tid & 31));
        const unsigned mask = warp_items >= 32 ? 0xffffffffu : ((1u << warp_items) - 1u);
        (void)mask;
        const int32_t h = item / VPR, c8 = item - h * VPR;
        int32_t cur_lp = -1, page = -1;
        int32_t cur_lq = -1;
        uint16_t* st = nullptr;  // statistics row of the open logical page (k_max; k_min + D)
        uint4 mx = make_uint4(0u, 0u, 0u, 0u), mn = mx;
        for (int32_t i = i_lo; i < i_hi; ++i) {
            const int32_t t = pos0 + i;
            uint4 kv, vv;
            if (single && i == 0 && item == tid) {
                kv = k0;
                vv = v0;
            } else {
                kv = *reinterpret_cast<const uint4*>(kb + i * tstride + (int64_t)item * 8);
                vv = *reinterpret_cast<const uint4*>(vb + i * tstride + (int64_t)item * 8);
            }
            const int32_t lp = t / P;
            if (lp != cur_lp) {
                cur_lp = lp;
                page = -1;
                if (lp >= L.max_pages_per_req) {
                    set_err(dev_err, DATTN_DEVERR_LEN_OOB);
                } else {
                    const int32_t pg = bt[lp];
                    if (pg < 0) set_err(dev_err, DATTN_DEVERR_UNMAPPED_PAGE);
                    else if (pg >= L.num_pages) set_err(dev_err, DATTN_DEVERR_PAGE_OOB);
                    else page = pg;
                }
            }
            if constexpr (FMT != DATTN_KV_BF16) {
                // every lane of a row takes part in the reductions, mapped page or not
                const float mk = row_absmax<VPR>(kv, mask), mv = row_absmax<VPR>(vv, mask);
                const bool i4 = FMT == DATTN_KV_INT4 || (FMT == DATTN_KV_MIXED && head_is_i4(hf, h));
                if (page >= 0) {
                    const int32_t slot = t - lp * P;
                    const int64_t row = ((int64_t)page * Hkv + h) * P + slot;  // the scales' row
                    // the codes' row: the mixed pool keeps each format in its own region
                    int64_t crow = row;
                    uint8_t* kd = k_code;
                    uint8_t* vd = v_code;
                    if constexpr (FMT == DATTN_KV_MIXED) {
                        const int32_t h4 = hf.h4, h8 = Hkv - h4;
                        crow = ((int64_t)page * (i4 ? h4 : h8) + head_class_index(hf, h, i4)) * P +
                               slot;
                        if (i4) {
                            const int64_t region8 = (int64_t)L.num_pages * h8 * P * D;
                            kd += region8;
                            vd += region8;
                        }
                    }
                    float ks, vs;
                    if (i4) {
                        const uint32_t kc = quant4_chunk(kv, mk, ks);
                        const uint32_t vc = quant4_chunk(vv, mv, vs);
                        *reinterpret_cast<uint32_t*>(kd + crow * (D / 2) + c8 * 4) = kc;
                        *reinterpret_cast<uint32_t*>(vd + crow * (D / 2) + c8 * 4) = vc;
                    } else {
                        const uint2 kc = quant8_chunk(kv, mk, ks);
                        const uint2 vc = quant8_chunk(vv, mv, vs);
                        *reinterpret_cast<uint2*>(kd + crow * D + c8 * 8) = kc;
                        *reinterpret_cast<uint2*>(vd + crow * D + c8 * 8) = vc;
                    }
                    if (c8 == 0) {  // [row / 16][K, V][row % 16]
                        float* sc = L.kv_scale + (row >> 4) * 32 + (row & 15);
                        sc[0] = ks;
                        sc[16] = vs;
                    }
                }
            } else if (page >= 0) {
                const int64_t dst = (((int64_t)page * Hkv + h) * P + (t - lp * P)) * D + c8 * 8;
                *reinterpret_cast<uint4*>(k_pool + dst) = kv;
                *reinterpret_cast<uint4*>(v_pool + dst) = vv;
            }
            if (stats == nullptr) continue;
            const int32_t lq = t >> 4;
            if (lq != cur_lq) {
                if (st != nullptr) {
                    *reinterpret_cast<uint4*>(st) = mx;
                    *reinterpret_cast<uint4*>(st + D) = mn;
                }
                cur_lq = lq;
                st = page >= 0
                    ? stats + (((int64_t)page * Hkv + h) * lpg + (t - lp * P) / 16) * 2 * D +
                          c8 * 8
                    : nullptr;
                if ((t & 15) == 0) {  // this append opens the logical page
                    mx = mn = kv;
                    continue;
                }
                if (st != nullptr) {
                    mx = *reinterpret_cast<const uint4*>(st);
                    mn = *reinterpret_cast<const uint4*>(st + D);
                }
            }
            bf16_fold8(kv, mx, mn);
        }
        if (st != nullptr) {
            *reinterpret_cast<uint4*>(st) = mx;
            *reinterpret_cast<uint4*>(st + D) = mn;
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

dattn_status_t launch_kv_append(const dattn_kv_layout& L, void* k_pool, void* v_pool,
                                uint16_t* stats, const uint16_t* k_new, const uint16_t* v_new,
                                int32_t B, int32_t T, int32_t* seq_lens, int32_t* dev_err,
                                cudaStream_t stream) {
    if (B == 0 || T == 0) return DATTN_OK;
    // a window of 64 aligned positions holds all T tokens whatever seq_lens % 16 is
    const bool single = T + 15 <= kAppendWindow;
    const int32_t nwin = single ? 1 : (T + 15 + kAppendWindow - 1) / kAppendWindow;
    const dim3 grid(nwin, B);
    const int32_t inplace = single ? 1 : 0;
    const int32_t items = L.num_kv_heads * (L.head_dim / 8);
    const dim3 block(min(kAppendMaxThreads, (items + 31) / 32 * 32));
    auto pick = [&](auto bf16, auto f8, auto i4, auto mix) {
        return L.kv_format == DATTN_KV_MIXED  ? mix
             : L.kv_format == DATTN_KV_INT4   ? i4
             : L.kv_format == DATTN_KV_FP8_E4M3 ? f8
                                                : bf16;
    };
    auto kern = L.head_dim == 64
                    ? pick(kv_append_kernel<64, DATTN_KV_BF16>, kv_append_kernel<64, DATTN_KV_FP8_E4M3>,
                           kv_append_kernel<64, DATTN_KV_INT4>, kv_append_kernel<64, DATTN_KV_MIXED>)
                    : pick(kv_append_kernel<128, DATTN_KV_BF16>,
                           kv_append_kernel<128, DATTN_KV_FP8_E4M3>,
                           kv_append_kernel<128, DATTN_KV_INT4>,
                           kv_append_kernel<128, DATTN_KV_MIXED>);
    KvHeadFormats hf;
    if (head_formats(L, hf) != DATTN_OK) return DATTN_ERR_INVALID_ARG;
    dattn_kv_layout Ld = L;
    Ld.head_format = nullptr;  // a host array: the kernel reads hf
    const cudaError_t e = launch_pdl(kern, grid, block, 0, stream, Ld, hf, k_pool, v_pool, stats,
                                     k_new, v_new, T, seq_lens, inplace, dev_err);
    if (e != cudaSuccess) return DATTN_ERR_CUDA;
    if (!single) {
        if (launch_pdl(advance_lengths_kernel, dim3((B + 255) / 256), dim3(256), 0, stream,
                       seq_lens, B, T) != cudaSuccess)
            return DATTN_ERR_CUDA;
    }
    return DATTN_OK;
}

}  // namespace dattn
