// gemm_mma.cu -- prefill Q8_0 x q8_0 GEMM on the warp-level int8 tensor
// instruction (mma.sync.m16n8k32.s8).
//
// Y[t][i] = sum_b d_w(i,b) * d_a(t,b) * isum(t,i,b)
//
// Each 32-wide k block is one q8_0 block on both operands, so one
// m16n8k32 instruction produces the exact int32 block dot products of a
// 16 x 8 tile, which are scaled by d_w * d_a (exact in f32) and accumulated
// in f32 once per block ("12 - r5-r6 re-ranking + structural rewrite spec",
// sec. 2 and 3.1: raw bytes staged by 16-byte async copies, values unpacked
// in registers at MMA time).  This is the legacy (pre-tcgen05) tensor path;
// it is kept as the exact baseline the tcgen05 kernel is measured against.
//
// CTA tile: 128 weight rows x 64 tokens, 8 blocks (k = 256) per stage,
// double-buffered; 8 warps in a 4 x 2 grid, 32 x 32 outputs per warp.
// Requires k/32 % 8 == 0 (every 8-block group of a weight row is 16-byte
// aligned); other shapes use the generic kernel.
#include "q8_common.cuh"

namespace {

constexpr int BM = 128, BN = 64, BKB = 8;
constexpr int kWRow = 272;   // 8 raw Q8_0 blocks per weight row per stage
constexpr int kARow = 272;   // 256 B of qs, padded by 16 B (bank spread)
constexpr int kDRow = 32;    // 8 ds words per token per stage
constexpr int kStageBytes = BM * kWRow + BN * kARow + BN * kDRow;  // 54272
constexpr int kThreads = 256;

__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool valid)
{
    const int sz = valid ? 16 : 0;  // 0 => zero-fill the 16 destination bytes
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(q8::smem_u32(dst)), "l"(src), "r"(sz)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_0() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void mma_s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                       uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(0), "r"(0), "r"(0), "r"(0));
}

// 4 qs bytes of a raw weight block starting at byte offset `o` (2-byte aligned)
__device__ __forceinline__ uint32_t ld_qs_word(const uint8_t *p, int o)
{
    const uint32_t *w = reinterpret_cast<const uint32_t *>(p + (o & ~3));
    return (o & 3) ? __byte_perm(w[0], w[1], 0x5432) : w[0];
}

__global__ void __launch_bounds__(kThreads)
gemm_mma_kernel(const uint8_t *__restrict__ w, int64_t n, int nb, const int8_t *__restrict__ qs,
                const uint32_t *__restrict__ ds, int64_t t, float *__restrict__ y)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wm = warp & 3, wn = warp >> 2;
    const int g = lane >> 2, c = lane & 3;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * BM;
    const int64_t t0 = static_cast<int64_t>(blockIdx.y) * BN;
    const int64_t pitch = static_cast<int64_t>(nb) * 34;
    const int64_t k = static_cast<int64_t>(nb) * 32;
    const int nkb = nb / BKB;

    auto load_stage = [&](int kb, int buf) {
        uint8_t *sw = smem + buf * kStageBytes;
        uint8_t *sa = sw + BM * kWRow;
        uint8_t *sd = sa + BN * kARow;
        for (int idx = tid; idx < BM * 17; idx += kThreads) {
            const int r = idx / 17, cc = idx - r * 17;
            const int64_t row = n0 + r;
            const bool ok = row < n;
            const uint8_t *src = w + (ok ? row : 0) * pitch + static_cast<int64_t>(kb) * kWRow + 16 * cc;
            cp_async16(sw + r * kWRow + 16 * cc, src, ok);
        }
        for (int idx = tid; idx < BN * 16; idx += kThreads) {
            const int r = idx >> 4, cc = idx & 15;
            const int64_t tok = t0 + r;
            const bool ok = tok < t;
            const int8_t *src = qs + (ok ? tok : 0) * k + static_cast<int64_t>(kb) * 256 + 16 * cc;
            cp_async16(sa + r * kARow + 16 * cc, src, ok);
        }
        for (int idx = tid; idx < BN * 2; idx += kThreads) {
            const int r = idx >> 1, cc = idx & 1;
            const int64_t tok = t0 + r;
            const bool ok = tok < t;
            const uint32_t *src = ds + (ok ? tok : 0) * nb + kb * BKB + 4 * cc;
            cp_async16(sd + r * kDRow + 16 * cc, src, ok);
        }
    };

    float acc[2][4][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][j][e] = 0.0f;

    load_stage(0, 0);
    cp_async_commit();
    for (int kb = 0; kb < nkb; ++kb) {
        if (kb + 1 < nkb) {
            load_stage(kb + 1, (kb + 1) & 1);
            cp_async_commit();
            cp_async_wait_1();
        } else {
            cp_async_wait_0();
        }
        __syncthreads();
        const uint8_t *sw = smem + (kb & 1) * kStageBytes;
        const uint8_t *sa = sw + BM * kWRow;
        const uint8_t *sd = sa + BN * kARow;
#pragma unroll 2
        for (int b = 0; b < BKB; ++b) {
            uint32_t af[2][4];
            float dw[2][2];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                const uint8_t *r0 = sw + (wm * 32 + mt * 16 + g) * kWRow;
                const uint8_t *r1 = r0 + 8 * kWRow;
                const int o = 34 * b + 2 + 4 * c;
                af[mt][0] = ld_qs_word(r0, o);
                af[mt][1] = ld_qs_word(r1, o);
                af[mt][2] = ld_qs_word(r0, o + 16);
                af[mt][3] = ld_qs_word(r1, o + 16);
                dw[mt][0] = __half2float(*reinterpret_cast<const __half *>(r0 + 34 * b));
                dw[mt][1] = __half2float(*reinterpret_cast<const __half *>(r1 + 34 * b));
            }
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
                const int tk = wn * 32 + nt * 8;
                const uint8_t *ar = sa + (tk + g) * kARow + 32 * b;
                const uint32_t b0 = *reinterpret_cast<const uint32_t *>(ar + 4 * c);
                const uint32_t b1 = *reinterpret_cast<const uint32_t *>(ar + 16 + 4 * c);
                const uint32_t dv0 = *reinterpret_cast<const uint32_t *>(sd + (tk + 2 * c) * kDRow + 4 * b);
                const uint32_t dv1 = *reinterpret_cast<const uint32_t *>(sd + (tk + 2 * c + 1) * kDRow + 4 * b);
                const float da0 = __half2float(__ushort_as_half(static_cast<unsigned short>(dv0 & 0xffffu)));
                const float da1 = __half2float(__ushort_as_half(static_cast<unsigned short>(dv1 & 0xffffu)));
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    int d[4];
                    mma_s8(d, af[mt][0], af[mt][1], af[mt][2], af[mt][3], b0, b1);
                    acc[mt][nt][0] = fmaf(dw[mt][0] * da0, static_cast<float>(d[0]), acc[mt][nt][0]);
                    acc[mt][nt][1] = fmaf(dw[mt][0] * da1, static_cast<float>(d[1]), acc[mt][nt][1]);
                    acc[mt][nt][2] = fmaf(dw[mt][1] * da0, static_cast<float>(d[2]), acc[mt][nt][2]);
                    acc[mt][nt][3] = fmaf(dw[mt][1] * da1, static_cast<float>(d[3]), acc[mt][nt][3]);
                }
            }
        }
        __syncthreads();
    }

    // C fragment: d0,d1 -> (row g, tokens 2c, 2c+1); d2,d3 -> (row g+8, ...)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int64_t r0 = n0 + wm * 32 + mt * 16 + g;
            const int64_t tk = t0 + wn * 32 + nt * 8 + 2 * c;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int64_t row = r0 + (e >> 1) * 8;
                const int64_t tok = tk + (e & 1);
                if (row < n && tok < t) y[tok * n + row] = acc[mt][nt][e];
            }
        }
}

} // namespace

namespace q8 {

int gemm_mma_launch(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, int64_t t, float *y,
                    cudaStream_t s)
{
    const int smem = 2 * kStageBytes;
    if (!set_max_dynamic_smem(reinterpret_cast<const void *>(gemm_mma_kernel), smem, 1)) return Q8_ERR_LAUNCH;
    const dim3 grid(static_cast<unsigned>((n + BM - 1) / BM), static_cast<unsigned>((t + BN - 1) / BN));
    gemm_mma_kernel<<<grid, kThreads, smem, s>>>(static_cast<const uint8_t *>(w), n, static_cast<int>(k / 32), qs,
                                                 ds, t, y);
    return launch_status();
}

} // namespace q8
