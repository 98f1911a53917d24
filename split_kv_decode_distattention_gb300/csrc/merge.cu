// Log-sum-exp aggregation of MicroAttention partials (dattn_merge).
//
// "Infinite-LLM: Efficient LLM Service for Long Context with DistAttention and Distributed
// KVCache", section "结果聚合与通信开销降低" (Fig. 4b): m_g = max_j m_j,
// e_g = sum_j e_j exp(m_j - m_g), Attention = sum_j MA_j exp(m_j - m_g) / e_g. The page
// notes that this aggregation costs under 1% of the MicroAttention work. Here one warp
// merges one (request, query head): lanes stride over the head dimension and loop over the
// chunks, and the chunk weights are computed once per chunk. A request's chunks are either a
// contiguous range of rows (chunk_indptr) or, for partials gathered from R ranks, the rows
// r B + b of the stacked [R][B] layout an all-gather leaves (dattn_merge_gathered).
#include "common.cuh"
#include "internal.h"

namespace dattn {

namespace {

constexpr int kMergeWarps = 4;

__global__ void __launch_bounds__(kMergeWarps * 32)
merge_kernel(int32_t B, int32_t C, int32_t Hq, int32_t D, const int32_t* __restrict__ indptr,
             int32_t R, const float* __restrict__ m, const float* __restrict__ e,
             const float* __restrict__ MA, float* __restrict__ out, float* __restrict__ m_g,
             float* __restrict__ e_g, float* __restrict__ MA_g, int32_t* dev_err) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    grid_dependency_wait();  // the partials may come from the previous kernel on the stream
    grid_launch_dependents();
    const int32_t b = blockIdx.x;
    const int32_t h = blockIdx.y * kMergeWarps + warp;
    if (h >= Hq) return;
    // chunk k of request b lives in row k (indptr) or in row k B + b (R gathered ranks)
    int32_t c0 = 0, c1 = R;
    if (indptr) {
        c0 = indptr[b];
        c1 = indptr[b + 1];
        if (c0 < 0 || c1 > C || c1 < c0) {
            if (lane == 0) set_err(dev_err, DATTN_DEVERR_CHUNK_OOB);
            c0 = min(max(c0, 0), C);
            c1 = min(max(c1, c0), C);
        }
    }
    auto row = [&](int32_t c) -> int64_t { return indptr ? (int64_t)c : (int64_t)c * B + b; };
    const float ninf = -__int_as_float(0x7f800000);
    float mg = ninf;
    for (int32_t c = c0 + lane; c < c1; c += 32) mg = fmaxf(mg, m[row(c) * Hq + h]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mg = fmaxf(mg, __shfl_xor_sync(0xffffffffu, mg, off));

    float acc[4] = {0.f, 0.f, 0.f, 0.f};  // D <= 128: lane owns d = lane + 32 * i
    float eg = 0.f;
    if (mg != ninf) {
        for (int32_t c = c0; c < c1; ++c) {
            const int64_t rc = row(c);
            const float mc = m[rc * Hq + h];
            if (mc == ninf) continue;  // an empty chunk adds nothing
            const float w = expf(mc - mg);
            eg += e[rc * Hq + h] * w;
            const float* ma = MA + (rc * Hq + h) * D;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (lane + 32 * i < D) acc[i] += ma[lane + 32 * i] * w;
        }
    }
    const int64_t o = ((int64_t)b * Hq + h) * D;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int d = lane + 32 * i;
        if (d >= D) continue;
        if (out) out[o + d] = eg > 0.f ? acc[i] / eg : 0.f;
        if (MA_g) MA_g[o + d] = acc[i];
    }
    if (lane == 0) {
        if (m_g) m_g[(int64_t)b * Hq + h] = mg;
        if (e_g) e_g[(int64_t)b * Hq + h] = eg;
    }
}

}  // namespace

dattn_status_t launch_merge(int32_t B, int32_t C, int32_t Hq, int32_t D, const int32_t* indptr,
                            int32_t R, const float* m, const float* e, const float* MA,
                            float* out, float* m_g, float* e_g, float* MA_g, int32_t* dev_err,
                            cudaStream_t stream) {
    if (B == 0 || Hq == 0) return DATTN_OK;
    const dim3 grid(B, (Hq + kMergeWarps - 1) / kMergeWarps);
    return launch_pdl(merge_kernel, grid, dim3(kMergeWarps * 32), 0, stream, B, C, Hq, D, indptr,
                      R, m, e, MA, out, m_g, e_g, MA_g, dev_err) == cudaSuccess
               ? DATTN_OK
               : DATTN_ERR_CUDA;
}

}  // namespace dattn
