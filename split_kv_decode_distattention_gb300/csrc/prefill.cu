// Block-sparse prefill (dattn_prefill): a chunk of Tq new query tokens per request attends
// the paged cache causally, key block by key block.
//
// "LLM长序列服务优化：LServe的块稀疏注意力技术": §2.1.1 cuts the KV history into fixed
// 64-token blocks and loads and computes only the chosen ones; §2.1.2 gives streaming heads a
// static Lambda pattern (the initial blocks plus the blocks next to the query) and retrieval
// heads a set of blocks chosen at run time; §2.2.1 walks the chosen blocks with a block
// iterator, so the compute loop has no branches on the mask.
//
// GB300 design. One CTA takes one 64-token query block of one query head (the g heads of a
// KV head are neighbouring CTAs, so their K/V reads meet in L2). A producer warp is the block
// iterator: it walks the head's key blocks for this query block and streams each block's four
// 16-token K and V row groups through an 8-stage shared-memory ring with 3-D TMA boxes (the
// decode's boxes and swizzle), issuing four tiles side by side, one lane each. Four consumer
// warps own 16 query rows each and take a whole key block per step: S = Q K^T on mma.sync
// m16n8k16 (bf16, fp32 accumulate; the query rows stay in shared memory), the causal and
// length mask, an online softmax in base 2 whose row sums stay per thread until the end, and
// O += P V with P taken straight from the S accumulators (as two bf16 terms). Every warp reads every stage, so a
// stage is released after four arrivals. No CTA depends on another: no workspace, no merge.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dattn {

namespace {

#define kPfNegInf (-__int_as_float(0x7f800000))

constexpr int kPfBlock = 64;                       // query and key block, tokens
constexpr int kPfWarps = 4;                        // consumer warps, 16 query rows each
constexpr int kPfThreads = (kPfWarps + 1) * 32;
constexpr int kPfStages = 8;                       // 16-token tiles in the ring: two key blocks
constexpr int kPfTiles = kPfBlock / 16;            // tiles per key block

struct PfParams {
    int32_t num_pages, Hkv, P, max_pages;
    const int32_t* block_table;
    const uint16_t* q;
    int32_t B, Tq, Hq, g;
    float sl2;  // scale * log2(e)
    const int32_t* seq_lens;
    int32_t nqb;  // query-block slots per (request, head): ceil(Tq / 64) + 1
    // block sparsity (head_kind == nullptr: dense causal)
    const int8_t* head_kind;
    int32_t sink_blocks, local_blocks, max_sel, qblock_stride;
    const int32_t* block_lists;
    float* out;
    float* m_out;
    float* e_out;
    int32_t* dev_err;
};

// Shared memory: the ring of stages (K tile, then V tile), each consumer warp's 16 query rows
// (in the K tiles' swizzled layout, read by ldmatrix), the full and empty barriers, the
// per-stage metadata (valid rows | skip flag) and the producer's compacted block ids.
struct PfSmem {
    uint32_t stage_bytes, stages, qs, bars, meta, comp, total;
};

__host__ __device__ inline PfSmem pf_smem_layout(int D) {
    PfSmem s;
    s.stage_bytes = 64u * (uint32_t)D;  // K and V: 16 rows of D bf16 each
    uint32_t o = 0;
    s.stages = o; o += kPfStages * s.stage_bytes;
    s.qs = o;     o += kPfWarps * 32u * (uint32_t)D;  // each warp's 16 query rows
    s.bars = o;   o += 2u * kPfStages * 8u;
    s.meta = o;   o += kPfStages * 4u;
    s.comp = o;   o += 32u * 4u;  // the producer's compacted block ids
    s.total = o + 1024u;  // slack to align the base to 1024 bytes (TMA swizzle)
    return s;
}

// The key blocks one (request, KV head) attends for query block qb, in the order the
// producer loads them: the block iterator of the head's kind.
struct BlockIter {
    int kind;
    int32_t qb, n;
    int32_t s_end, l0;          // streaming: sinks [0, s_end), band [l0, qb]
    const int32_t* list;        // retrieval: the row of block_lists
    __device__ int32_t count() const { return n; }
    // the i-th entry (i < n): a key block, or -1 for a retrieval entry that is not a block at
    // or before qb. Both the producer and the consumers skip the -1 entries the same way:
    // 32 entries at a time, a ballot of the valid ones, then those blocks in order.
    __device__ int32_t at(int32_t i) const {
        if (kind == DATTN_HEAD_STREAMING) return i < s_end ? i : l0 + (i - s_end);
        if (kind == DATTN_HEAD_RETRIEVAL) {
            const int32_t kb = __ldg(list + i);
            return (kb >= 0 && kb <= qb) ? kb : -1;
        }
        return i;
    }
};

__device__ __forceinline__ BlockIter make_iter(const PfParams& p, int32_t b, int32_t kvh,
                                               int32_t qb) {
    BlockIter it;
    it.qb = qb;
    it.kind = p.head_kind ? p.head_kind[kvh] : DATTN_HEAD_DENSE;
    if (it.kind < 0 || it.kind > 2) it.kind = DATTN_HEAD_DENSE;
    it.list = nullptr;
    it.s_end = it.l0 = 0;
    if (it.kind == DATTN_HEAD_STREAMING) {
        it.s_end = min(max(p.sink_blocks, 0), qb + 1);
        it.l0 = max(it.s_end, qb - p.local_blocks + 1);
        it.n = it.s_end + max(0, qb + 1 - it.l0);
    } else if (it.kind == DATTN_HEAD_RETRIEVAL) {
        it.list = p.block_lists + (((int64_t)b * p.Hkv + kvh) * p.qblock_stride + qb) * p.max_sel;
        it.n = p.max_sel;
    } else {
        it.n = qb + 1;
    }
    return it;
}

constexpr int32_t kPfSkip = 1 << 16;  // stage metadata: no data in this stage

__device__ __forceinline__ uint64_t policy_evict_normal() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

template <int D>
__global__ void __launch_bounds__(kPfThreads, 2)
prefill_kernel(const __grid_constant__ PfParams p, const __grid_constant__ CUtensorMap tmap_k,
               const __grid_constant__ CUtensorMap tmap_v) {
    constexpr int KS = D / 16;  // k-steps of Q K^T
    constexpr int NT = D / 8;   // n-tiles (8 channels) of P V
    extern __shared__ uint8_t smem_raw[];
    __shared__ int abort_flag;
    uint8_t* base;
    {  // align by the shared-window offset: the TMA swizzle pattern is defined on it
        const uint32_t off = smem_u32(smem_raw);
        base = smem_raw + (((off + 1023u) & ~1023u) - off);
    }
    const PfSmem L = pf_smem_layout(D);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // CTA -> (request, query-block slot, query head): the heads of one query block are
    // neighbours, and a request's last query blocks (the most key blocks) start first.
    int32_t c = blockIdx.x;
    const int32_t h = c % p.Hq;
    c /= p.Hq;
    const int32_t j = p.nqb - 1 - c % p.nqb;
    const int32_t b = c / p.nqb;
    const uint32_t bars = smem_u32(base + L.bars);
    int32_t* meta = reinterpret_cast<int32_t*>(base + L.meta);
    volatile int* abort_p = &abort_flag;
    if (tid == 0) {
        for (int s = 0; s < kPfStages; ++s) {
            mbar_init(bars + 8u * s, 1);
            mbar_init(bars + 8u * (kPfStages + s), kPfWarps);
        }
        *abort_p = 0;
        fence_mbar_init();
    }
    if (warp == kPfWarps && lane == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    grid_dependency_wait();  // the lengths and the pool may come from the previous kernel
    grid_launch_dependents();
    __syncthreads();

    const int32_t Ln = p.seq_lens[b];
    if (Ln < p.Tq || Ln > p.max_pages * p.P) {
        if (tid == 0 && h == 0 && j == 0) set_err(p.dev_err, DATTN_DEVERR_LEN_OOB);
        return;
    }
    const int32_t c0 = Ln - p.Tq;  // position of the chunk's first token
    const int32_t qb = c0 / kPfBlock + j;
    const int32_t p_lo = max(c0, qb * kPfBlock), p_hi = min(Ln, qb * kPfBlock + kPfBlock);
    if (p_lo >= p_hi) return;  // no query of the chunk in this slot
    const int32_t kvh = h / p.g;
    const BlockIter it = make_iter(p, b, kvh, qb);
    if (it.kind == DATTN_HEAD_RETRIEVAL && qb >= p.qblock_stride) {
        if (tid == 0) set_err(p.dev_err, DATTN_DEVERR_LEN_OOB);
        return;
    }
    const int32_t nblk = it.count();

    if (warp == kPfWarps) {
        // -------------------------------------------------- producer warp: the block iterator
        const uint64_t pol = policy_evict_normal();  // later query blocks read the same K/V
        const uint32_t tile_bytes = 32u * (uint32_t)D;
        const uint32_t stages0 = smem_u32(base + L.stages);
        int32_t* comp = reinterpret_cast<int32_t*>(base + L.comp);
        int32_t k = 0;  // tiles issued: tile k uses stage k % kPfStages
        bool stop = false;
        for (int32_t i0 = 0; i0 < nblk && !stop; i0 += 32) {
            const int32_t kbl = i0 + lane < nblk ? it.at(i0 + lane) : -1;
            const unsigned vm = __ballot_sync(0xffffffffu, kbl >= 0);
            if (kbl >= 0) comp[__popc(vm & ((1u << lane) - 1u))] = kbl;
            __syncwarp();
            const int32_t nv = __popc(vm);
            for (int32_t v0 = 0; v0 < nv && !stop; v0 += 32 / kPfTiles) {
                // resolve up to 8 blocks (32 tiles): lane l takes tile l % 4 of block v0 + l / 4
                const int32_t nb = min(32 / kPfTiles, nv - v0);
                int32_t y = 0, lohi = kPfSkip;
                if (lane < nb * kPfTiles) {
                    const int32_t kb = comp[v0 + lane / kPfTiles];
                    const int32_t t0 = kb * kPfBlock + 16 * (lane % kPfTiles);
                    if (t0 < p_hi) {  // keys after the last query are never visible
                        const int32_t lp = t0 / p.P;
                        const int32_t page = __ldg(p.block_table + (int64_t)b * p.max_pages + lp);
                        if (page < 0) {
                            set_err(p.dev_err, DATTN_DEVERR_UNMAPPED_PAGE);
                        } else if (page >= p.num_pages) {
                            set_err(p.dev_err, DATTN_DEVERR_PAGE_OOB);
                        } else {
                            y = (page * p.Hkv + kvh) * p.P + (t0 - lp * p.P);
                            lohi = min(16, Ln - t0);
                        }
                    }
                }
                // issue a block at a time, lane u of the group taking tile u
                for (int32_t bi = 0; bi < nb; ++bi, k += kPfTiles) {
                    const int32_t src = min(bi * kPfTiles + lane, 31);
                    const int32_t ty = __shfl_sync(0xffffffffu, y, src);
                    const int32_t tm = __shfl_sync(0xffffffffu, lohi, src);
                    bool ok = true;
                    if (lane < kPfTiles) {
                        const int32_t kk = k + lane, stg = kk % kPfStages;
                        if (kk >= kPfStages)
                            ok = mbar_wait(bars + 8u * (kPfStages + stg),
                                           ((kk / kPfStages) - 1) & 1, abort_p, p.dev_err);
                        if (ok) {
                            const uint32_t full = bars + 8u * stg;
                            meta[stg] = tm;
                            if (tm & kPfSkip) {
                                mbar_arrive(full);
                            } else {
                                mbar_arrive_expect_tx(full, 2u * tile_bytes);
                                const uint32_t dst = stages0 + (uint32_t)stg * L.stage_bytes;
                                tma_load_3d(dst, &tmap_k, 0, ty, 0, full, pol);
                                tma_load_3d(dst + tile_bytes, &tmap_v, 0, ty, 0, full, pol);
                            }
                        }
                    }
                    if (__any_sync(0xffffffffu, !ok)) {
                        stop = true;
                        break;
                    }
                }
            }
            __syncwarp();  // comp is rewritten for the next 32 entries
        }
        // after an abort, wait (bounded in total) for copies still in flight
        if (lane == 0 && *abort_p) {
            const unsigned long long t0 = global_timer_ns();
            for (int32_t kk = max(0, k - kPfStages); kk < k; ++kk) {
                while (!mbar_try_wait(bars + 8u * (kk % kPfStages), (kk / kPfStages) & 1) &&
                       global_timer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
        return;
    }

    // -------------------------------------------------- consumer warps: 16 query rows each
    const int g8 = lane >> 2, tig = lane & 3;
    const int32_t pos0 = qb * kPfBlock + warp * 16 + g8, pos1 = pos0 + 8;  // query positions
    const bool ok0 = pos0 >= p_lo && pos0 < p_hi, ok1 = pos1 >= p_lo && pos1 < p_hi;
    const bool all_rows = p_lo == qb * kPfBlock && p_hi == qb * kPfBlock + kPfBlock;
    // The warp's 16 query rows go to shared memory once, in the K tiles' swizzled layout
    // ([half][row][64 values]); each k-step reads them as mma A fragments with ldmatrix, which
    // leaves the registers to the accumulator.
    const uint32_t qbase = smem_u32(base + L.qs) + (uint32_t)warp * 32u * (uint32_t)D;
    for (int idx = lane; idx < 16 * (D / 8); idx += 32) {
        const int r = idx / (D / 8), ch = idx - r * (D / 8);
        const int32_t pos = qb * kPfBlock + warp * 16 + r;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (pos >= p_lo && pos < p_hi)
            v = __ldg(reinterpret_cast<const uint4*>(
                p.q + (((int64_t)b * p.Tq + (pos - c0)) * p.Hq + h) * D) + ch);
        *reinterpret_cast<uint4*>(base + (qbase - smem_u32(base)) + (ch >> 3) * 2048u +
                                  swz128((uint32_t)r, (uint32_t)(ch & 7))) = v;
    }
    __syncwarp();
    const uint32_t qrow = (lane & 7) + (((lane >> 3) & 1) << 3), qcs = lane >> 4;
    float o[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m0 = kPfNegInf, m1 = kPfNegInf, l0 = 0.f, l1 = 0.f;  // row max (base 2), partial sums
    const uint32_t stage0 = smem_u32(base + L.stages);
    // ldmatrix lane addresses. K (B of S = Q K^T): matrices (keys 0-7 | 8-15) x (chunk
    // 2ks | 2ks + 1) give b0, b1 of both 8-key n-tiles. V (B of O = P V, transposed):
    // matrices (keys 0-7 | 8-15) x (chunk c | c + 1) give b0, b1 of n-tiles c and c + 1.
    const uint32_t krow = (lane & 7) + ((lane >> 4) << 3), kcs = (lane >> 3) & 1;
    const uint32_t vrow = (lane & 7) + (((lane >> 3) & 1) << 3), vcs = lane >> 4;
    int32_t k = 0;
    bool aborted = false;
    for (int32_t i0 = 0; i0 < nblk && !aborted; i0 += 32) {
      const int32_t kbl = i0 + lane < nblk ? it.at(i0 + lane) : -1;
      unsigned vm = __ballot_sync(0xffffffffu, kbl >= 0);
      for (; vm != 0u; vm &= vm - 1u, k += kPfTiles) {
        const int32_t kb = __shfl_sync(0xffffffffu, kbl, __ffs(vm) - 1);
        bool ok = true;
#pragma unroll
        for (int u = 0; u < kPfTiles; ++u)
            ok = ok && mbar_wait(bars + 8u * ((k + u) % kPfStages), ((k + u) / kPfStages) & 1,
                                 abort_p, p.dev_err);
        if (!__all_sync(0xffffffffu, ok)) {
            aborted = true;
            break;
        }
        const bool diag = kb == qb;  // only the diagonal block needs the causal test
        int32_t hi[kPfTiles];
        bool full_tiles = true;  // every tile holds 16 valid keys
#pragma unroll
        for (int u = 0; u < kPfTiles; ++u) {
            const int32_t mt = meta[(k + u) % kPfStages];
            hi[u] = (mt & kPfSkip) ? -1 : mt;  // valid rows of the tile; -1: no data
            full_tiles = full_tiles && hi[u] == 16;
        }
        // warp-uniform: only the diagonal block, a short tile or a partly filled query block
        // needs the per-element mask
        const bool masked = diag || !full_tiles || !all_rows;
        // The block's four tiles go two at a time (32 keys), which keeps the scores of a half
        // in registers next to the query fragments and the accumulator.
#pragma unroll
        for (int hb = 0; hb < kPfTiles / 2; ++hb) {
        // ---- S = Q K^T over 32 keys (each query fragment serves both tiles) ---------------
        float s[2][2][4];
#pragma unroll
        for (int uu = 0; uu < 2; ++uu)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[uu][0][e] = s[uu][1][e] = 0.f;
        const bool t0ok = hi[2 * hb] >= 0, t1ok = hi[2 * hb + 1] >= 0;  // warp-uniform
        if (t0ok || t1ok) {
            const uint32_t kb0 = stage0 + (uint32_t)((k + 2 * hb) % kPfStages) * L.stage_bytes;
            const uint32_t kb1 = stage0 + (uint32_t)((k + 2 * hb + 1) % kPfStages) * L.stage_bytes;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const uint32_t qchunk = 2u * ks + qcs, chunk = 2u * ks + kcs;
                const uint32_t koff = (chunk >> 3) * 2048u + swz128(krow, chunk & 7u);
                uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
                ldsm_x4(qbase + (qchunk >> 3) * 2048u + swz128(qrow, qchunk & 7u), a0, a1, a2, a3);
                if (t0ok) {
                    ldsm_x4(kb0 + koff, b0, b1, b2, b3);
                    mma_bf16(s[0][0], a0, a1, a2, a3, b0, b1);
                    mma_bf16(s[0][1], a0, a1, a2, a3, b2, b3);
                }
                if (t1ok) {
                    ldsm_x4(kb1 + koff, b0, b1, b2, b3);
                    mma_bf16(s[1][0], a0, a1, a2, a3, b0, b1);
                    mma_bf16(s[1][1], a0, a1, a2, a3, b2, b3);
                }
            }
        }
        // ---- mask (length, causal, empty tiles), scale to base 2, row maxima -------------
        float mx0 = kPfNegInf, mx1 = kPfNegInf;
#pragma unroll
        for (int uu = 0; uu < 2; ++uu) {
            const int u = 2 * hb + uu;
#pragma unroll
            for (int n = 0; n < 2; ++n) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (masked) {
                        const int32_t r = 8 * n + 2 * tig + (e & 1);  // key row within the tile
                        const int32_t key = kb * kPfBlock + 16 * u + r;
                        const bool row1 = e >= 2;
                        bool v = r < hi[u] && (row1 ? ok1 : ok0);
                        if (diag) v = v && key <= (row1 ? pos1 : pos0);
                        s[uu][n][e] = v ? s[uu][n][e] * p.sl2 : kPfNegInf;
                    } else {
                        s[uu][n][e] *= p.sl2;
                    }
                }
                mx0 = fmaxf(mx0, fmaxf(s[uu][n][0], s[uu][n][1]));
                mx1 = fmaxf(mx1, fmaxf(s[uu][n][2], s[uu][n][3]));
            }
        }
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        // ---- online softmax ---------------------------------------------------------------
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float mu0 = mn0 == kPfNegInf ? 0.f : mn0, mu1 = mn1 == kPfNegInf ? 0.f : mn1;
        if (__any_sync(0xffffffffu, mn0 != m0 || mn1 != m1)) {
            const float al0 = exp2f(m0 - mu0), al1 = exp2f(m1 - mu1);
            l0 *= al0;
            l1 *= al1;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                o[nt][0] *= al0; o[nt][1] *= al0; o[nt][2] *= al1; o[nt][3] *= al1;
            }
        }
        m0 = mn0;
        m1 = mn1;
#pragma unroll
        for (int uu = 0; uu < 2; ++uu) {
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                s[uu][n][0] = exp2f(s[uu][n][0] - mu0);
                s[uu][n][1] = exp2f(s[uu][n][1] - mu0);
                s[uu][n][2] = exp2f(s[uu][n][2] - mu1);
                s[uu][n][3] = exp2f(s[uu][n][3] - mu1);
                l0 += s[uu][n][0] + s[uu][n][1];
                l1 += s[uu][n][2] + s[uu][n][3];
            }
        }
        // ---- O += P V, one 16-key step per tile; P is the S accumulator in A layout -------
#pragma unroll
        for (int uu = 0; uu < 2; ++uu) {
            const int u = 2 * hb + uu;
            if (hi[u] < 0) continue;  // warp-uniform
            // P as two bf16 terms (hi + lo: 16 significant bits), as the decode takes it
            const uint32_t a0 = pack_bf16(s[uu][0][0], s[uu][0][1]);
            const uint32_t a1 = pack_bf16(s[uu][0][2], s[uu][0][3]);
            const uint32_t a2 = pack_bf16(s[uu][1][0], s[uu][1][1]);
            const uint32_t a3 = pack_bf16(s[uu][1][2], s[uu][1][3]);
            const uint32_t e0 = pack_bf16(s[uu][0][0] - bf16_lo(a0), s[uu][0][1] - bf16_hi(a0));
            const uint32_t e1 = pack_bf16(s[uu][0][2] - bf16_lo(a1), s[uu][0][3] - bf16_hi(a1));
            const uint32_t e2 = pack_bf16(s[uu][1][0] - bf16_lo(a2), s[uu][1][1] - bf16_hi(a2));
            const uint32_t e3 = pack_bf16(s[uu][1][2] - bf16_lo(a3), s[uu][1][3] - bf16_hi(a3));
            // V rows past the length hold stale data: zero them so that 0 * stale stays 0
            uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
            if (hi[u] < 16) {
                const int t0 = 2 * tig, t1 = 2 * tig + 1;
                mlo = (t0 < hi[u] ? 0x0000ffffu : 0u) | (t1 < hi[u] ? 0xffff0000u : 0u);
                mhi = (t0 + 8 < hi[u] ? 0x0000ffffu : 0u) | (t1 + 8 < hi[u] ? 0xffff0000u : 0u);
            }
            const uint32_t vbase = stage0 + (uint32_t)((k + u) % kPfStages) * L.stage_bytes +
                                   32u * (uint32_t)D;
#pragma unroll
            for (int nt = 0; nt < NT; nt += 2) {
                const uint32_t chunk = (uint32_t)nt + vcs;
                uint32_t b0, b1, b2, b3;
                ldsm_x4_trans(vbase + (chunk >> 3) * 2048u + swz128(vrow, chunk & 7u), b0, b1, b2,
                              b3);
                if (hi[u] < 16) {  // warp-uniform
                    b0 &= mlo;
                    b1 &= mhi;
                    b2 &= mlo;
                    b3 &= mhi;
                }
                mma_bf16(o[nt], a0, a1, a2, a3, b0, b1);
                mma_bf16(o[nt], e0, e1, e2, e3, b0, b1);
                mma_bf16(o[nt + 1], a0, a1, a2, a3, b2, b3);
                mma_bf16(o[nt + 1], e0, e1, e2, e3, b2, b3);
            }
        }
        }  // half of the block
        __syncwarp();
        if (lane == 0) {
#pragma unroll
            for (int u = 0; u < kPfTiles; ++u)
                mbar_arrive(bars + 8u * (kPfStages + (k + u) % kPfStages));
        }
      }
    }
    // ---- epilogue: row sums across the four lanes of a row, then out = O / l -------------
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const bool okr = half ? ok1 : ok0;
        if (!okr) continue;
        const int32_t pos = half ? pos1 : pos0;
        const int64_t row = ((int64_t)b * p.Tq + (pos - c0)) * p.Hq + h;
        const float inv = half ? inv1 : inv0;
        float* orow = p.out + row * D;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            *reinterpret_cast<float2*>(orow + 8 * nt + 2 * tig) =
                make_float2(o[nt][2 * half] * inv, o[nt][2 * half + 1] * inv);
        if (tig == 0) {
            const float m = half ? m1 : m0;
            if (p.m_out) p.m_out[row] = m == kPfNegInf ? kPfNegInf : m * kLn2;
            if (p.e_out) p.e_out[row] = half ? l1 : l0;
        }
    }
}

std::mutex g_pf_mutex;
int g_pf_smem_set[2] = {0, 0};

template <int D>
dattn_status_t launch_prefill_d(const PfParams& p, const void* k_pool, const void* v_pool,
                                int64_t ctas, cudaStream_t stream) {
    const PfSmem L = pf_smem_layout(D);
    {
        std::lock_guard<std::mutex> lock(g_pf_mutex);
        int& set = g_pf_smem_set[D == 128 ? 1 : 0];
        if ((int)L.total > set) {
            if (cudaFuncSetAttribute(prefill_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)L.total) != cudaSuccess)
                return DATTN_ERR_CUDA;
            set = (int)L.total;
        }
    }
    alignas(64) CUtensorMap tk;
    alignas(64) CUtensorMap tv;
    const int64_t rows = (int64_t)p.num_pages * p.Hkv * p.P;
    dattn_status_t st;
    if ((st = make_kv_tensor_map(&tk, k_pool, rows, D)) != DATTN_OK) return st;
    if ((st = make_kv_tensor_map(&tv, v_pool, rows, D)) != DATTN_OK) return st;
    if (launch_pdl(prefill_kernel<D>, dim3((unsigned)ctas), dim3(kPfThreads), L.total, stream, p,
                   tk, tv) != cudaSuccess)
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
        return layout->kv_format == DATTN_KV_FP8_E4M3 ? DATTN_ERR_UNSUPPORTED
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
    return layout->head_dim == 64 ? launch_prefill_d<64>(p, k_pool, v_pool, ctas, s)
                                  : launch_prefill_d<128>(p, k_pool, v_pool, ctas, s);
}
