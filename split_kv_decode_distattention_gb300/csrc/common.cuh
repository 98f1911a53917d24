// Device-side building blocks shared by the dattn kernels (sm_103a).
//
// This header holds the inline-PTX wrappers (mbarrier, TMA tensor and bulk copies, ldmatrix,
// mma.sync, movmatrix), the bounded pipeline wait, and the balanced split plan.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dattn.h"

namespace dattn {

// ------------------------------------------------------------------ balanced split plan
// The tiles of all segments are laid end to end: W tiles in total. CTA c of G covers
// [floor(c*W/G), floor((c+1)*W/G)). Tile t belongs to CTA ceil((t+1)*G/W) - 1. The pieces
// that one segment leaves in the CTAs from c_first to c_last get workspace slots c + s,
// which are distinct for distinct (CTA, segment) pairs. Callers keep W < 2^40 and
// G < 2^20, so every product fits in 64 bits.
__host__ __device__ inline int64_t split_begin(int64_t W, int32_t G, int32_t c) {
    return W * (int64_t)c / (int64_t)G;
}
__host__ __device__ inline int32_t split_owner(int64_t t, int64_t W, int32_t G) {
    return (int32_t)(((t + 1) * (int64_t)G - 1) / W);
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned long long kWaitLimitNs = 5ull * 1000ull * 1000ull * 1000ull;  // 5 s

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete, for at most kWaitLimitNs. A wait
// that runs out sets *abort and the TIMEOUT bit of the error word. Once *abort is set, every
// later wait returns false at once, so the CTA drains through its barriers instead of
// hanging. Returns true when the phase completed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          int32_t* dev_err) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_timer_ns();
    while (true) {
        if (*abort) return false;
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            if (dev_err) atomicOr(dev_err, DATTN_DEVERR_TIMEOUT);
            return false;
        }
    }
}

// Atomic add at GPU scope with acquire-release semantics; returns the old value.
__device__ __forceinline__ int32_t atom_add_acq_rel_gpu(int32_t* ptr, int32_t v) {
    int32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
                 : "=r"(old)
                 : "l"(ptr), "r"(v)
                 : "memory");
    return old;
}

// Warms L2 with [ptr, ptr + bytes): thread gt of gthreads prefetches every gthreads-th
// 128-byte line. A prefetch returns no data, so it may run before the dependency wait even
// for data the previous kernel writes (L2 is where those writes land).
__device__ __forceinline__ void prefetch_l2_range(const void* ptr, size_t bytes, int64_t gt,
                                                  int64_t gthreads) {
    const char* c = static_cast<const char*>(ptr);
    for (size_t off = (size_t)gt * 128u; off < bytes; off += (size_t)gthreads * 128u)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(c + off));
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 3-D tiled TMA load: box at (x, y, z) into shared memory, completing on mbarrier bar.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                            int32_t z, uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

// 2-D tiled TMA load: box at (x, y) into shared memory, completing on mbarrier bar.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int32_t x, int32_t y,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// Bulk copy global -> shared (both 16-byte aligned, bytes a multiple of 16), completing on
// the barrier's transaction count, with an L2 policy for the source.
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A(16x16, row) * B(16x8, col) + D, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
        "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The four E4M3 codes of x (byte i = code i) as two fp16x2 words: lo = codes 0, 1 and
// hi = codes 2, 3, the lower code in the lower half. Every E4M3 value is an fp16 value, so
// the conversion is exact.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t x, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(x));
}

// E4M3 codes of four floats (rounded to nearest even, saturated to +-448), code i in byte i.
__device__ __forceinline__ uint32_t f32x4_to_e4m3(float a0, float a1, float a2, float a3) {
    uint32_t lo, hi;
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\tcvt.u32.u16 %0, t;\n\t}"
        : "=r"(lo)
        : "f"(a0), "f"(a1));
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\tcvt.u32.u16 %0, t;\n\t}"
        : "=r"(hi)
        : "f"(a2), "f"(a3));
    return lo | (hi << 16);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float f16_lo(uint32_t v) {
    return __low2float(*reinterpret_cast<const __half2*>(&v));
}
__device__ __forceinline__ float f16_hi(uint32_t v) {
    return __high2float(*reinterpret_cast<const __half2*>(&v));
}

// Transpose of an 8x8 b16 matrix held one row-pair per thread (mma fragment layout).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Byte offset of 16-byte chunk `chunk` of row `row` in a [rows][128 B] box written by TMA
// with CU_TENSOR_MAP_SWIZZLE_128B (the box base is 1024-byte aligned).
__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t chunk) {
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a [rows][64 B] box written by TMA
// with CU_TENSOR_MAP_SWIZZLE_64B (the box base is 512-byte aligned).
__device__ __forceinline__ uint32_t swz64(uint32_t row, uint32_t chunk) {
    return row * 64u + ((chunk ^ ((row >> 1) & 3u)) << 4);
}

// 2^x by the special-function unit (ex2.approx.ftz: relative error near 2^-22, subnormal results
// flushed to +0, 2^-inf = +0)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a [rows][32 B] box written by TMA
// with CU_TENSOR_MAP_SWIZZLE_32B (the box base is 256-byte aligned).
__device__ __forceinline__ uint32_t swz32(uint32_t row, uint32_t chunk) {
    return row * 32u + ((chunk ^ ((row >> 2) & 1u)) << 4);
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a [rows][RB bytes] box written by TMA
// with the swizzle of that row size.
template <uint32_t RB>
__device__ __forceinline__ uint32_t swz_rows(uint32_t row, uint32_t chunk) {
    static_assert(RB == 128 || RB == 64 || RB == 32, "swizzled rows are 32, 64 or 128 bytes");
    return RB == 128 ? swz128(row, chunk) : RB == 64 ? swz64(row, chunk) : swz32(row, chunk);
}

// The 4-bit codes at nibble K of each 16-bit half of x (bits 4K..4K+3 and 16+4K..16+4K+3,
// each code stored as n = code + 8) as two fp16 subnormals: nibbles 0 and 2 (2 and 3 are first
// shifted down by 8 bits, one shift serving both) masked in place are n * 2^-24, nibbles 1
// and 3 are 16 n * 2^-24. Every value is exact; the factor 16 and the offset 8 are taken out
// by the caller (the query of an odd nibble is divided by 16, and 8 times the sum of the
// other operand is subtracted from the products).
template <int K>
__device__ __forceinline__ uint32_t i4pair_raw(uint32_t x) {
    const uint32_t y = K >= 2 ? x >> 8 : x;
    return y & ((K & 1) == 0 ? 0x000f000fu : 0x00f000f0u);
}

// Programmatic dependent launch: a kernel launched with programmatic stream serialization may
// start while the previous kernel on the stream is still running. It must wait here before it
// reads anything that kernel writes. Without a programmatic launch this returns at once.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next programmatically launched kernel on the stream be scheduled early.
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- row quantization of the 8-bit and 4-bit pools (the append and the fused append) ----
// A row of d bf16 values is handled 8 channels (one 16-byte chunk) per lane, the lanes of a
// row consecutive. scale = max|x| / 448 (8-bit) or / 7 (4-bit), each code from x / scale, both
// divisions in IEEE fp32.

__device__ __forceinline__ float bf(uint32_t h) { return __uint_as_float(h << 16); }

// Max |x| of the 8 bf16 values of a 16-byte chunk.
__device__ __forceinline__ float absmax8(const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        m = fmaxf(m, fmaxf(fabsf(bf(w[i] & 0xffffu)), fabsf(bf(w[i] >> 16))));
    return m;
}

// E4M3 codes of the 8 bf16 values of a chunk divided by s (s > 0), code i in byte i.
__device__ __forceinline__ uint2 quant8(const uint4& v, float s) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    float x[8];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[2 * i] = __fdiv_rn(bf(w[i] & 0xffffu), s);
        x[2 * i + 1] = __fdiv_rn(bf(w[i] >> 16), s);
    }
    return make_uint2(f32x4_to_e4m3(x[0], x[1], x[2], x[3]), f32x4_to_e4m3(x[4], x[5], x[6], x[7]));
}

// Max |x| of a row, from this lane's 8-channel chunk; `mask` holds the lanes of this warp in
// the loop, and the VPR lanes of a row are consecutive and all in it.
template <int VPR>
__device__ __forceinline__ float row_absmax(const uint4& v, unsigned mask) {
    float m = absmax8(v);
#pragma unroll
    for (int off = 1; off < VPR; off <<= 1) m = fmaxf(m, __shfl_xor_sync(mask, m, off));
    return m;
}

// 8-bit row scale (row max |x| = m) and the E4M3 codes of one chunk.
__device__ __forceinline__ uint2 quant8_chunk(const uint4& v, float m, float& scale) {
    scale = __fdiv_rn(m, 448.0f);
    return scale > 0.f ? quant8(v, scale) : make_uint2(0u, 0u);
}

// 4-bit codes of the 8 bf16 values of a chunk divided by s (s > 0): code c + 8 of channel
// 2j in the low nibble of byte j, of channel 2j + 1 in its high nibble.
__device__ __forceinline__ uint32_t quant4(const uint4& v, float s) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int c0 = min(7, max(-7, __float2int_rn(__fdiv_rn(bf(w[i] & 0xffffu), s))));
        const int c1 = min(7, max(-7, __float2int_rn(__fdiv_rn(bf(w[i] >> 16), s))));
        out |= (uint32_t)((c0 + 8) | ((c1 + 8) << 4)) << (8 * i);
    }
    return out;
}

// 4-bit row scale (row max |x| = m) and the packed codes of one chunk.
__device__ __forceinline__ uint32_t quant4_chunk(const uint4& v, float m, float& scale) {
    scale = __fdiv_rn(m, 7.0f);
    return scale > 0.f ? quant4(v, scale) : 0x88888888u;
}


// Folds 8 bf16 key channels (one 16-byte chunk) into a logical page's running k_max / k_min,
// per channel with strict comparisons, so that on a tie the earlier value stays.
__device__ __forceinline__ void bf16_fold8(const uint4& k, uint4& mx, uint4& mn) {
    const uint32_t kw[4] = {k.x, k.y, k.z, k.w};
    uint32_t xw[4] = {mx.x, mx.y, mx.z, mx.w};
    uint32_t nw[4] = {mn.x, mn.y, mn.z, mn.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t a = kw[i] & 0xffffu, z = kw[i] >> 16;
        uint32_t x0 = xw[i] & 0xffffu, x1 = xw[i] >> 16;
        uint32_t n0 = nw[i] & 0xffffu, n1 = nw[i] >> 16;
        if (bf16_lo(a) > bf16_lo(x0)) x0 = a;
        if (bf16_lo(a) < bf16_lo(n0)) n0 = a;
        if (bf16_lo(z) > bf16_lo(x1)) x1 = z;
        if (bf16_lo(z) < bf16_lo(n1)) n1 = z;
        xw[i] = x0 | (x1 << 16);
        nw[i] = n0 | (n1 << 16);
    }
    mx = make_uint4(xw[0], xw[1], xw[2], xw[3]);
    mn = make_uint4(nw[0], nw[1], nw[2], nw[3]);
}

__device__ __forceinline__ void st_shared_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint32_t a, uint32_t b) {
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4& v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void set_err(int32_t* dev_err, int32_t bit) {
    if (dev_err) atomicOr(dev_err, bit);
}

}  // namespace dattn
