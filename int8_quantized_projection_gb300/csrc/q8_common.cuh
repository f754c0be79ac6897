// q8_common.cuh -- internal helpers of libq8proj (not part of the C ABI).
//
// PTX wrappers for sm_103a (mbarrier, bulk/TMA copies, globaltimer), the
// status plumbing shared by every translation unit, and the register-level
// q8_0 block encoder used by all three quantizing kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/q8proj.h"

#define Q8_FULL_MASK 0xffffffffu

// A bounded on-device wait gives up after this many nanoseconds, records
// Q8_ERR_DEVICE_TIMEOUT in the translation unit's error word and lets the
// kernel return instead of hanging the GPU.
#ifndef Q8_WAIT_LIMIT_NS
#define Q8_WAIT_LIMIT_NS 1000000000ull
#endif
// Waits that let a kernel's own copies (and tensor-core work) in flight land
// before it exits -- on the normal path and after another wait gave up -- have
// a limit of their own, so that a build with a short main-loop limit still
// never exits with a copy writing into its shared memory.
#ifndef Q8_DRAIN_LIMIT_NS
#define Q8_DRAIN_LIMIT_NS 1000000000ull
#endif

namespace q8 {

// ---------------------------------------------------------------------------
// host-side helpers (defined in abi.cu)
// ---------------------------------------------------------------------------
int device_sm_count();                 // cached per device; 0 on error
bool device_is_sm103();                // current device is compute capability 10.3
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
int launch_status();                   // Q8_OK or Q8_ERR_LAUNCH from cudaGetLastError
// Raise a kernel's dynamic shared-memory limit once per (device, slot);
// slots are small integers owned by the calling translation unit.
bool set_max_dynamic_smem(const void *func, int bytes, int slot);

// Launch `kernel` with programmatic dependent launch allowed: it may start
// while the previous kernel on the stream is still running, so it must call
// griddep_wait() before touching memory that kernel may write.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) != cudaSuccess) return Q8_ERR_LAUNCH;
    return launch_status();
}

// The same with thread-block clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
int launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster_x,
                       Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster_x);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) != cudaSuccess) return Q8_ERR_LAUNCH;
    return launch_status();
}

// Host: a 2-D tiled TMA tensor map (element type dt, dims {d0 (inner), d1},
// row stride in bytes, box {b0, b1}, out-of-bounds elements read as zero),
// encoded through the driver entry point (abi.cu).  False on failure.
bool make_map_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, uint64_t d0, uint64_t d1,
                 uint64_t stride_bytes, uint32_t b0, uint32_t b1, CUtensorMapSwizzle sw);

// The same in three dimensions: dims {d0, d1, d2}, byte strides of
// dimensions 1 and 2, box {b0, b1, b2}.
bool make_map_3d(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                 CUtensorMapSwizzle sw);

// Per-translation-unit device error words are read and cleared through these
// (each .cu file that has bounded waits defines one).
int gemv_take_error(cudaStream_t s);
int gemv_generic_launch(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, float *y,
                        int64_t tokens, cudaStream_t s);
// small-batch kernel (gemv.cu): 1 <= tokens <= Q8_GEMV_MAX_TOKENS, (k/32) % 8 == 0
int gemv_small_launch(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, float *y,
                      int64_t tokens, cudaStream_t s);
int gemv_small_grouped_launch(const q8_gemv_proj *projs, int count, int64_t k, const int8_t *qs, const uint32_t *ds,
                              int64_t tokens, cudaStream_t s);
// Token counts up to kSlicedMaxTokens run the small-batch kernel over 16-token
// slices of the plane (each slice streams the weights once more): up to four
// passes cost less than the GEMM's weight pre-pass and its f16 re-read.
constexpr int64_t kSlicedMaxTokens = 64;
int gemv_sliced_launch(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, float *y,
                       int64_t tokens, cudaStream_t s);
// small-batch kernel (gemv.cu) for asymmetric 4-bit blocks: 1 <= tokens <= 16, (k/32) % 8 == 0
int gemv_small_q4a_launch(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, float *y,
                          int64_t tokens, cudaStream_t s);
int gemv_small_q4a_grouped_launch(const q8_gemv_proj *projs, int count, int64_t k, const int8_t *qs,
                                  const uint32_t *ds, int64_t tokens, cudaStream_t s);
// staged batch-1 kernel (gemv.cu) for asymmetric 4-bit blocks: k % 128 == 0,
// k / 128 <= kGemvStagedMaxChunks (the activation is staged in shared memory)
constexpr int kGemvStagedMaxChunks = 512;
int gemv_staged_q4a_launch(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, float *y,
                           cudaStream_t s);
int gemm_take_error(cudaStream_t s);
int quant_take_error(cudaStream_t s);

// ---------------------------------------------------------------------------
// device-side PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete; false if the wait
// ran past `limit_ns`.  A limit of 0 (a build that gives up at once) makes
// the wait one non-blocking test.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns = Q8_WAIT_LIMIT_NS)
{
    if (limit_ns == 0) return mbar_test_wait(bar, parity);
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// Bulk (non-tensor) copy global -> shared, completion counted in bytes on
// `bar`.  src, dst 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Wait until the previous kernel on the stream has finished and its writes
// are visible (no-op when launched without programmatic dependent launch).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel on the stream to begin launching.
__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c)
{
    return __dp4a(static_cast<int>(a), static_cast<int>(b), c);
}

// 2-D tiled TMA load of one box into shared memory at dst, completing on the
// mbarrier at bar (shared addresses); x is the inner coordinate in elements.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int x, int y, int z, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// Four int8 codes (one 32-bit word) -> two f16x2 words, exactly: byte b
// becomes the f16 1024 + (b ^ 0x80), minus 1152.  lo holds bytes 0 and 1
// (byte 0 in the low half), hi bytes 2 and 3.
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t q, uint32_t &lo, uint32_t &hi)
{
    const uint32_t x = q ^ 0x80808080u;
    const uint32_t l = __byte_perm(x, 0x64646464u, 0x5140);
    const uint32_t h = __byte_perm(x, 0x64646464u, 0x5342);
    const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));  // 1152
    const __half2 lv = __hsub2(*reinterpret_cast<const __half2 *>(&l), bias);
    const __half2 hv = __hsub2(*reinterpret_cast<const __half2 *>(&h), bias);
    lo = *reinterpret_cast<const uint32_t *>(&lv);
    hi = *reinterpret_cast<const uint32_t *>(&hv);
}

// ---------------------------------------------------------------------------
// q8_0 encoder: one 32-element block held by 8 consecutive lanes, 4 values
// per lane (lane & 7 == 0 holds elements 0..3).  Every lane of the warp must
// call it (full-mask shuffles); lanes whose group is out of range simply
// discard the result.  Steps as in the quantize body of "54 - r51 -
// producer-fused A-quantize mode 1", sec. 3.2: block amax, d = amax/127 in
// f32, di = 1/d (0 when d = 0), q = rint(x*di) clamped to +-127, ssum = sum q,
// d stored as f16 (round to nearest even).  Division, reciprocal and product
// are the IEEE round-to-nearest forms, so the codes are a pure function of
// the f32 inputs.
// ---------------------------------------------------------------------------
struct Q8Enc {
    uint32_t qword;  // 4 int8 codes of this lane, little-endian
    uint32_t dsword; // f16(d) | ssum << 16 (same value on all 8 lanes)
};

__device__ __forceinline__ int clamp127(int v) { return max(-127, min(127, v)); }

// The scalar steps of the q8_0 encoding of one block: d = amax / 127 and its
// reciprocal (both IEEE round-to-nearest), a code = rni(v * 1/d) clamped to
// +-127, and the packed d | ssum word.  amax and ssum do not depend on the
// order they are reduced in (a maximum; an integer sum).
__device__ __forceinline__ float q8_block_d(float amax) { return __fdiv_rn(amax, 127.0f); }
__device__ __forceinline__ float q8_block_di(float d) { return (d != 0.0f) ? __frcp_rn(d) : 0.0f; }
__device__ __forceinline__ int q8_code(float v, float di) { return clamp127(__float2int_rn(__fmul_rn(v, di))); }

// Whether the clamp in q8_code can change a code of this block.  When d is
// a normal float (or 0, infinite or NaN) every |v| <= amax gives
// |v * di| <= 127 (1 + 2^-24)^2 / (1 - 2^-24) < 127.5 (three round-to-nearest
// steps, each within 2^-24), so rint(v * di) already lies in [-127, 127], and
// a non-finite product converts to 0 either way.  Only a subnormal d (amax
// below 127 * 2^-126), where d carries fewer significant bits, can push a
// code past 127.
__device__ __forceinline__ bool q8_block_needs_clamp(float d) { return d > 0.0f && d < 1.17549435e-38f; }

// q8_code for a block whose d does not need the clamp (the same code).
__device__ __forceinline__ int q8_code_unclamped(float v, float di) { return __float2int_rn(__fmul_rn(v, di)); }
__device__ __forceinline__ uint32_t q8_dsword(float d, int ssum)
{
    return static_cast<uint32_t>(__half_as_ushort(__float2half_rn(d))) |
           (static_cast<uint32_t>(static_cast<uint16_t>(static_cast<int16_t>(ssum))) << 16);
}

// Four codes (each in [-127, 127]) packed little-endian into a word: the low
// byte of each, by byte permutes.
__device__ __forceinline__ uint32_t pack4(int a, int b, int c, int d)
{
    const uint32_t ab = __byte_perm(static_cast<uint32_t>(a), static_cast<uint32_t>(b), 0x0040u);  // a0 b0 . .
    const uint32_t cd = __byte_perm(static_cast<uint32_t>(c), static_cast<uint32_t>(d), 0x0040u);  // c0 d0 . .
    return __byte_perm(ab, cd, 0x5410u);                                                          // a0 b0 c0 d0
}

// Codes rounded on the FMA pipe.  p = fma(x, 1/d, +0) is the f32 product
// rounded once (IEEE: adding +0 changes no non-zero result, and a compiler
// may not drop it, since it turns a -0 product into +0), and p + 1.5 * 2^23
// rounded to f32 is rint(p), ties to even, for |p| < 2^22: the sum lies
// where the f32 spacing is 1.  Its bits are 0x4B400000 + rint(p): the low
// byte is the code and the wrapped sum of the bits gives the code sum.
// Because p comes from an FMA, the add cannot be fused with the multiply
// (which would round the exact product instead: another code where p is
// exactly k + 0.5).
constexpr float kRoundMagic = 12582912.0f;
constexpr uint32_t kRoundMagicBits = 0x4B400000u;

__device__ __forceinline__ void round_by_add2(float a, float b, float di, uint32_t &ba, uint32_t &bb)
{
    const float2 p = __ffma2_rn(make_float2(a, b), make_float2(di, di), make_float2(0.0f, 0.0f));
    const float2 r = __fadd2_rn(p, make_float2(kRoundMagic, kRoundMagic));
    ba = __float_as_uint(r.x);
    bb = __float_as_uint(r.y);
}

// Whether a block's codes may be rounded by the add: d is 0 (every product
// is +-0) or a normal finite float (every |p| < 127.5, as for the unclamped
// codes).  A subnormal or non-finite d takes the clamped codes.
__device__ __forceinline__ bool block_rounds_by_add(float d)
{
    return d == 0.0f || (d >= 1.17549435e-38f && d <= 3.40282347e+38f);
}

// 8 adjacent lanes hold one 32-element block, a float4 each.
__device__ __forceinline__ Q8Enc q8_encode8(float4 v)
{
    float a = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    a = fmaxf(a, __shfl_xor_sync(Q8_FULL_MASK, a, 1));
    a = fmaxf(a, __shfl_xor_sync(Q8_FULL_MASK, a, 2));
    a = fmaxf(a, __shfl_xor_sync(Q8_FULL_MASK, a, 4));
    const float d = q8_block_d(a);
    const float di = q8_block_di(d);
    int s;
    Q8Enc e;
    if (block_rounds_by_add(d)) {  // the codes' low bytes straight from the rounded sums' bits
        uint32_t b0, b1, b2, b3;
        round_by_add2(v.x, v.y, di, b0, b1);
        round_by_add2(v.z, v.w, di, b2, b3);
        s = static_cast<int>(b0 + b1 + b2 + b3 - 4u * kRoundMagicBits);
        e.qword = __byte_perm(__byte_perm(b0, b1, 0x0040u), __byte_perm(b2, b3, 0x0040u), 0x5410u);
    } else {
        const int q0 = q8_code(v.x, di);
        const int q1 = q8_code(v.y, di);
        const int q2 = q8_code(v.z, di);
        const int q3 = q8_code(v.w, di);
        s = q0 + q1 + q2 + q3;
        e.qword = (static_cast<uint32_t>(q0) & 0xffu) | ((static_cast<uint32_t>(q1) & 0xffu) << 8) |
                  ((static_cast<uint32_t>(q2) & 0xffu) << 16) | (static_cast<uint32_t>(q3) << 24);
    }
    s += __shfl_xor_sync(Q8_FULL_MASK, s, 1);
    s += __shfl_xor_sync(Q8_FULL_MASK, s, 2);
    s += __shfl_xor_sync(Q8_FULL_MASK, s, 4);
    e.dsword = q8_dsword(d, s);
    return e;
}

// The 32 lanes of a warp hold one block, a value each: this lane's code,
// and the block's d | ssum word (the same on every lane).
__device__ __forceinline__ int q8_encode32(float v, uint32_t &dsword)
{
    float a = fabsf(v);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) a = fmaxf(a, __shfl_xor_sync(Q8_FULL_MASK, a, o));
    const float d = q8_block_d(a);
    const int q = q8_code(v, q8_block_di(d));
    int s = q;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) s += __shfl_xor_sync(Q8_FULL_MASK, s, o);
    dsword = q8_dsword(d, s);
    return q;
}

// Producer arithmetic, one implementation for the standalone producers
// (quantize.cu) and the activation staging of the fused GEMV (gemv.cu), so
// both compute the same f32 bits and therefore the same plane.
//
// SwiGLU element: silu(g) * u with the hardware exp2 and reciprocal (a few
// ulp).  For g < -87.3 the denominator exceeds 2^126 and the quotient is 0,
// where the true value is below 1e-36.
__device__ __forceinline__ float silu_mul(float g, float u)
{
    return __fmul_rn(__fdividef(g, __fadd_rn(1.0f, __expf(-g))), u);
}

__device__ __forceinline__ float4 silu_mul4(float4 g, float4 u)
{
    return make_float4(silu_mul(g.x, u.x), silu_mul(g.y, u.y), silu_mul(g.z, u.z), silu_mul(g.w, u.w));
}

// RMSNorm.  A row's sum of squares is accumulated by P threads: thread p
// adds the squares of float4 p, p + P, ..., p + (J-1)P in that order with
// fused multiply-adds, each warp sums its 32 partials by xor shuffles
// (16, 8, 4, 2, 1), and the P/32 warp sums are added in warp order.
// (J, P) depend only on d and on max_p, the most threads a row may take.
__device__ __forceinline__ float rms_sumsq4(float ss, float4 v)
{
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    return fmaf(v.w, v.w, ss);
}

__device__ __forceinline__ float rms_warp_sum(float ss)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(Q8_FULL_MASK, ss, o);
    return ss;
}

__device__ __forceinline__ float rms_scale(float total, int d, float eps)
{
    return rsqrtf(total / static_cast<float>(d) + eps);
}

// y = (x * scale) * w, two roundings per element
__device__ __forceinline__ float4 rms_apply4(float4 v, float scale, float4 w)
{
    return make_float4(__fmul_rn(__fmul_rn(v.x, scale), w.x), __fmul_rn(__fmul_rn(v.y, scale), w.y),
                       __fmul_rn(__fmul_rn(v.z, scale), w.z), __fmul_rn(__fmul_rn(v.w, scale), w.w));
}

// float4 per thread (J, a power of two up to 16) and threads per row (P, a
// multiple of 32) for a row of F float4 with at most max_p threads.
__host__ __device__ inline void rms_row_mapping(int F, int max_p, int &J, int &P)
{
    J = 1;
    while (J < 16 && (F + J - 1) / J > max_p) J *= 2;
    P = ((F + J - 1) / J + 31) / 32 * 32;
}

// The most threads a row of the standalone RMSNorm takes: 512 when every CTA
// has at most one row (rows_pad <= the SM count, e.g. a decode token), else
// 256 (several rows per CTA, four CTAs per SM).
constexpr int kRmsMaxThreadsOneRow = 512;
constexpr int kRmsMaxThreadsManyRows = 256;

} // namespace q8
