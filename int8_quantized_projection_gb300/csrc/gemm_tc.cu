// gemm_tc.cu -- prefill Q8_0 x q8_0 GEMM on the 5th-generation tensor cores
// (tcgen05.mma, TMA, tensor memory).
//
// Y[t][i] = sum_b d_w(i,b) * d_a(t,b) * isum(t,i,b)
//
// sm_103a has no int8 kind of tcgen05.mma, so the int8 codes are widened to
// f16 (exact: |q| <= 127) and multiplied with kind::f16 into an f32 TMEM
// accumulator.  One MMA pair covers exactly one 32-wide q8_0 block, whose
// partial sums are integers of magnitude <= 32*127*127 < 2^24, so the tensor
// core returns the exact int32 block dot products.  Each block's result is
// then scaled by d_w * d_a (exact in f32) and added to an f32 register
// accumulator -- the per-block scale correction of "12 - r5-r6 re-ranking +
// structural rewrite spec" (sec. 2: raw bytes staged by bulk copies, values
// unpacked at MMA time) and the q8_0 plane of "54 - r51 - producer-fused
// A-quantize mode 1" (sec. 2.1).
//
// One CTA computes a 128 (weight rows) x 128 (tokens) tile over all of k.
// Warp roles (512 threads):
//   warp 0      TMA producer: raw Q8_0 rows (2D u16 map, 8 blocks per stage),
//               plane qs (2D u8 map, 128B swizzle) and ds words (2D u32 map)
//   warp 1      TMEM allocator and single-thread MMA issuer
//   warps 2-7   converters: raw int8 -> f16 operand tiles in the canonical
//               K-major no-swizzle layout, one 32-wide block at a time, plus
//               the block's scales as f32 (weight rows read with three
//               16-byte loads, bank-conflict free)
//   warps 8-15  epilogue: two warps per TMEM lane quarter, 64 tokens each;
//               per block, tcgen05.ld of the partial, acc += (d_w * d_a) *
//               partial with packed f32x2 multiply / fma, then one coalesced
//               store of Y
// Every mbarrier wait is bounded; a wait that runs out sets the CTA abort
// flag and the library error word, and all roles drain and exit.
#include <cuda.h>

#include "q8_common.cuh"

namespace {

__device__ unsigned int g_gemm_err;

constexpr int BM = 128, BN = 128;
constexpr int kBlocksPerStage = 8;                 // k = 256 per raw stage
constexpr int kRawStages = 2;
constexpr int kF16Slots = 4;
constexpr int kAcc = 4;                            // TMEM block buffers of BN columns
constexpr int kTmemCols = kAcc * BN;               // 512
constexpr int kConvThreads = 192;                  // warps 2-7
constexpr int kEpiThreads = 256;                   // warps 8-15
constexpr int kThreads = 64 + kConvThreads + kEpiThreads;  // 512

constexpr int kARawBytes = BM * 272;               // 34816
constexpr int kBRawHalf = BN * 128;                // 16384 (128B-swizzled rows)
constexpr int kBRawBytes = 2 * kBRawHalf;          // 32768
constexpr int kDRawBytes = BN * 32;                // 4096
constexpr int kStageTx = kARawBytes + kBRawBytes + kDRawBytes;  // 71680
constexpr int kF16Tile = 128 * 64;                 // 8192: 128 rows x 32 f16
constexpr int kF16SlotBytes = 2 * kF16Tile;        // A and B

// shared-memory map (offsets from a 1024-byte aligned base)
constexpr int OFF_BRAW = 0;                                        // 2 x 32768 (1024-aligned)
constexpr int OFF_ARAW = OFF_BRAW + kRawStages * kBRawBytes;       // 65536
constexpr int OFF_DRAW = OFF_ARAW + kRawStages * kARawBytes;       // 135168
constexpr int OFF_F16 = OFF_DRAW + kRawStages * kDRawBytes;        // 143360
constexpr int OFF_SCALE = OFF_F16 + kF16Slots * kF16SlotBytes;     // 208896
constexpr int OFF_BAR = OFF_SCALE + kAcc * 2 * 128 * 4;            // 212992
constexpr int kNumBars = 2 * kRawStages + 2 * kF16Slots + 4 * kAcc + 1; // 29 (last: MMA drain)
constexpr int OFF_MISC = OFF_BAR + kNumBars * 8;
constexpr int kSmemBytes = OFF_MISC + 16 + 1024;                   // + alignment slack

// ---------------------------------------------------------------------------
// PTX wrappers specific to this kernel
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// 32 consecutive TMEM columns of this warp's 32 lanes -> 32 registers per thread.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor, K-major, no swizzle: core matrices of
// 8 rows x 16 bytes; LBO = byte step between core matrices along k, SBO =
// byte step between 8-row groups.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3fffu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3fffu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3fffu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
    return d;                             // base offset 0, swizzle none
}

// Instruction descriptor: D f32, A and B f16, both K-major, M = 128, N = BN.
constexpr uint32_t kIdesc = (1u << 4) | (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);

// int8 x4 (one 32-bit word) -> two f16x2 words, exactly: byte b becomes the
// f16 1024 + (b ^ 0x80), minus 1152.
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

__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(20000u)  // suspend up to 20 us per try instead of spinning
        : "memory");
    return ok != 0;
}

// Bounded wait shared by all roles: gives up on the CTA abort flag or after
// the time limit (then raises the flag and the error word).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag)
{
    if (try_wait(bar, parity)) return true;
    const uint64_t t0 = q8::globaltimer_ns();
    for (;;) {
        if (try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (q8::globaltimer_ns() - t0 > Q8_WAIT_LIMIT_NS) {
            *abort_flag = 1;
            atomicOr(&g_gemm_err, 1u);
            return false;
        }
    }
}

// Wait that ignores the abort flag (used to drain in-flight async work
// before exit); still bounded.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = q8::globaltimer_ns();
    while (!try_wait(bar, parity)) {
        if (q8::globaltimer_ns() - t0 > Q8_WAIT_LIMIT_NS) {
            atomicOr(&g_gemm_err, 1u);
            return;
        }
    }
}

__device__ __forceinline__ void arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Converter step for weight row r, raw block BETA of the stage: read the 48
// bytes (three 16-byte aligned, bank-conflict-free loads) that contain the
// row's 34-byte block, write the 32 codes as f16 into the A tile and d as f32.
template <int BETA>
__device__ __forceinline__ void convert_a_row(const uint8_t *arow, uint8_t *a16, float *sw, int r)
{
    constexpr int off = 34 * BETA;
    constexpr int c0 = off >> 4;        // first 16-byte chunk
    constexpr int o = off & 15;         // block start within it (even)
    uint32_t w[12];
#pragma unroll
    for (int c = 0; c < 3; ++c) {
        const uint4 v = *reinterpret_cast<const uint4 *>(arow + 16 * (c0 + c));
        w[4 * c + 0] = v.x;
        w[4 * c + 1] = v.y;
        w[4 * c + 2] = v.z;
        w[4 * c + 3] = v.w;
    }
    const uint32_t dbits = (o & 2) ? (w[o >> 2] >> 16) : (w[o >> 2] & 0xffffu);
    sw[r] = __half2float(__ushort_as_half(static_cast<unsigned short>(dbits)));
    uint32_t qw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int ob = o + 2 + 4 * i;   // compile-time after unrolling
        qw[i] = (ob & 3) ? __byte_perm(w[ob >> 2], w[(ob >> 2) + 1], 0x5432) : w[ob >> 2];
    }
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) {
        uint4 v;
        i8x4_to_f16x4(qw[2 * kc], v.x, v.y);
        i8x4_to_f16x4(qw[2 * kc + 1], v.z, v.w);
        *reinterpret_cast<uint4 *>(a16 + (r >> 3) * 512 + kc * 128 + (r & 7) * 16) = v;
    }
}

// Converter step for one (token, 16-byte half-block) task of raw block BETA.
template <int BETA>
__device__ __forceinline__ void convert_b_task(const uint8_t *braw_stage, const uint8_t *draw_stage, uint8_t *b16,
                                               float *sa, int id)
{
    const int l = id & 31;
    const int tok = 16 * (id >> 5) + (l & 7) + 8 * (l >> 4);
    const int h = (l >> 3) & 1;
    constexpr int hh = BETA >> 2, bq = BETA & 3;
    const int c16 = 2 * bq + h;
    const uint8_t *braw = braw_stage + hh * kBRawHalf;
    const uint4 v = *reinterpret_cast<const uint4 *>(braw + tok * 128 + ((c16 ^ (tok & 7)) << 4));
    uint4 o0, o1;
    i8x4_to_f16x4(v.x, o0.x, o0.y);
    i8x4_to_f16x4(v.y, o0.z, o0.w);
    i8x4_to_f16x4(v.z, o1.x, o1.y);
    i8x4_to_f16x4(v.w, o1.z, o1.w);
    uint8_t *dst = b16 + (tok >> 3) * 512 + (tok & 7) * 16 + (2 * h) * 128;
    *reinterpret_cast<uint4 *>(dst) = o0;
    *reinterpret_cast<uint4 *>(dst + 128) = o1;
    if (h == 0) {
        const uint32_t dw = *reinterpret_cast<const uint32_t *>(draw_stage + tok * 32 + 4 * BETA);
        sa[tok] = __half2float(__ushort_as_half(static_cast<unsigned short>(dw & 0xffffu)));
    }
}

struct Bars {
    uint32_t b0;
    __device__ uint32_t raw_full(int s) const { return b0 + 8u * s; }
    __device__ uint32_t raw_empty(int s) const { return b0 + 8u * (kRawStages + s); }
    __device__ uint32_t f16_full(int s) const { return b0 + 8u * (2 * kRawStages + s); }
    __device__ uint32_t f16_empty(int s) const { return b0 + 8u * (2 * kRawStages + kF16Slots + s); }
    __device__ uint32_t acc_full(int s) const { return b0 + 8u * (2 * kRawStages + 2 * kF16Slots + s); }
    __device__ uint32_t acc_empty(int s) const { return b0 + 8u * (2 * kRawStages + 2 * kF16Slots + kAcc + s); }
    __device__ uint32_t sc_full(int s) const { return b0 + 8u * (2 * kRawStages + 2 * kF16Slots + 2 * kAcc + s); }
    __device__ uint32_t sc_empty(int s) const { return b0 + 8u * (2 * kRawStages + 2 * kF16Slots + 3 * kAcc + s); }
    __device__ uint32_t drain() const { return b0 + 8u * (kNumBars - 1); }
};

// One 32-wide block of the stage for the converter role.
template <int BETA>
__device__ __forceinline__ bool convert_block(const Bars &B, uint8_t *sm, float *scales, int s, int c,
                                              volatile int *abort_flag)
{
    const int slot = s % kRawStages;
    const int j = s * kBlocksPerStage + BETA;
    constexpr int fs = BETA % kF16Slots, sc = BETA % kAcc;
    if (BETA == 0 && !wait_bar(B.raw_full(slot), static_cast<uint32_t>(s / kRawStages) & 1u, abort_flag))
        return false;
    if (!wait_bar(B.f16_empty(fs), (static_cast<uint32_t>(j / kF16Slots) & 1u) ^ 1u, abort_flag)) return false;
    if (!wait_bar(B.sc_empty(sc), (static_cast<uint32_t>(j / kAcc) & 1u) ^ 1u, abort_flag)) return false;
    uint8_t *a16 = sm + OFF_F16 + fs * kF16SlotBytes;
    uint8_t *b16 = a16 + kF16Tile;
    float *sw = scales + sc * 256;
    float *sa = sw + 128;
    const uint8_t *braw = sm + OFF_BRAW + slot * kBRawBytes;
    const uint8_t *draw = sm + OFF_DRAW + slot * kDRawBytes;
    if (c < 128) {
        convert_a_row<BETA>(sm + OFF_ARAW + slot * kARawBytes + c * 272, a16, sw, c);
        convert_b_task<BETA>(braw, draw, b16, sa, c);
    } else {
        convert_b_task<BETA>(braw, draw, b16, sa, 128 + (c - 128));
        convert_b_task<BETA>(braw, draw, b16, sa, 192 + (c - 128));
    }
    q8::fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
    arrive(B.f16_full(fs));
    arrive(B.sc_full(sc));
    if (BETA == kBlocksPerStage - 1) arrive(B.raw_empty(slot));
    return true;
}

__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmD, int64_t n, int64_t t, int nb, float *__restrict__ y)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = q8::smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t *sm = smem_raw + (base - raw_base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Bars B{base + OFF_BAR};
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_MISC);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_MISC + 4);
    float *scales = reinterpret_cast<float *>(sm + OFF_SCALE);  // [kAcc][2][128]: d_w rows, d_a tokens

    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * BM;
    const int64_t t0 = static_cast<int64_t>(blockIdx.y) * BN;
    const int nstages = nb / kBlocksPerStage;

    if (threadIdx.x == 0) {
        *abort_flag = (*reinterpret_cast<volatile unsigned int *>(&g_gemm_err) != 0u) ? 1 : 0;
        uint64_t *b = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
        for (int s = 0; s < kRawStages; ++s) {
            q8::mbar_init(b + s, 1);                               // raw_full: TMA bytes
            q8::mbar_init(b + kRawStages + s, kConvThreads);       // raw_empty
        }
        for (int s = 0; s < kF16Slots; ++s) {
            q8::mbar_init(b + 2 * kRawStages + s, kConvThreads);   // f16_full
            q8::mbar_init(b + 2 * kRawStages + kF16Slots + s, 1);  // f16_empty: tcgen05.commit
        }
        uint64_t *a = b + 2 * kRawStages + 2 * kF16Slots;
        for (int s = 0; s < kAcc; ++s) {
            q8::mbar_init(a + s, 1);                     // acc_full: tcgen05.commit
            q8::mbar_init(a + kAcc + s, kEpiThreads);    // acc_empty
            q8::mbar_init(a + 2 * kAcc + s, kConvThreads); // sc_full
            q8::mbar_init(a + 3 * kAcc + s, kEpiThreads);  // sc_empty
        }
        q8::mbar_init(b + kNumBars - 1, 1);              // MMA drain
        q8::fence_mbar_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         q8::smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    q8::griddep_launch_dependents();
    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            // Inputs may come from the previous kernel on the stream; every other
            // role only touches data this thread brings in, and Y is written
            // after the last MMA, so this is the only wait needed.
            q8::griddep_wait();
            int issued = 0;
            for (int s = 0; s < nstages && !*abort_flag; ++s) {
                const int slot = s % kRawStages;
                const uint32_t use = static_cast<uint32_t>(s / kRawStages);
                if (!wait_bar(B.raw_empty(slot), (use & 1u) ^ 1u, abort_flag)) break;
                asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(B.raw_full(slot)),
                             "r"(kStageTx)
                             : "memory");
                tma_load_2d(base + OFF_ARAW + slot * kARawBytes, &tmA, s * 136, static_cast<int>(n0), B.raw_full(slot));
                tma_load_2d(base + OFF_BRAW + slot * kBRawBytes, &tmB, s * 256, static_cast<int>(t0), B.raw_full(slot));
                tma_load_2d(base + OFF_BRAW + slot * kBRawBytes + kBRawHalf, &tmB, s * 256 + 128,
                            static_cast<int>(t0), B.raw_full(slot));
                tma_load_2d(base + OFF_DRAW + slot * kDRawBytes, &tmD, s * 8, static_cast<int>(t0), B.raw_full(slot));
                issued = s + 1;
            }
            // drain: the last stages issued must have landed before the CTA exits
            for (int s = issued - kRawStages < 0 ? 0 : issued - kRawStages; s < issued; ++s)
                drain_bar(B.raw_full(s % kRawStages), static_cast<uint32_t>(s / kRawStages) & 1u);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            for (int j = 0; j < nb; ++j) {
                const int fs = j % kF16Slots, ab = j % kAcc;
                if (!wait_bar(B.f16_full(fs), static_cast<uint32_t>(j / kF16Slots) & 1u, abort_flag)) break;
                if (!wait_bar(B.acc_empty(ab), (static_cast<uint32_t>(j / kAcc) & 1u) ^ 1u, abort_flag)) break;
                tc_fence_after();
                const uint32_t a_addr = base + OFF_F16 + fs * kF16SlotBytes;
                const uint32_t b_addr = a_addr + kF16Tile;
                const uint32_t d = tmem + static_cast<uint32_t>(ab * BN);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)  // two K=16 steps = one 32-wide block
                    tc_mma_f16(d, smem_desc(a_addr + 256 * kk, 128, 512), smem_desc(b_addr + 256 * kk, 128, 512),
                               kIdesc, kk);
                tc_commit(B.f16_empty(fs));
                tc_commit(B.acc_full(ab));
            }
            // drain: every MMA issued must have completed before TMEM is freed
            tc_commit(B.drain());
            drain_bar(B.drain(), 0);
        }
    } else if (warp < 8) {
        // ------------------------------------------------------------ converters
        const int c = threadIdx.x - 64;  // 0..191
        for (int s = 0; s < nstages && !*abort_flag; ++s) {
            if (!convert_block<0>(B, sm, scales, s, c, abort_flag)) break;
            if (!convert_block<1>(B, sm, scales, s, c, abort_flag)) break;
            if (!convert_block<2>(B, sm, scales, s, c, abort_flag)) break;
            if (!convert_block<3>(B, sm, scales, s, c, abort_flag)) break;
            if (!convert_block<4>(B, sm, scales, s, c, abort_flag)) break;
            if (!convert_block<5>(B, sm, scales, s, c, abort_flag)) break;
            if (!convert_block<6>(B, sm, scales, s, c, abort_flag)) break;
            if (!convert_block<7>(B, sm, scales, s, c, abort_flag)) break;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;            // TMEM lane quarter of this warp
        const int hcol = (warp - 8) >> 2;  // column half: tokens [64*hcol, 64*hcol + 64)
        const int r = 32 * q + lane;       // tile row = TMEM lane
        float2 acc[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = make_float2(0.0f, 0.0f);
        bool ok = true;
        for (int j = 0; j < nb; ++j) {
            const int ab = j % kAcc;
            if (!wait_bar(B.acc_full(ab), static_cast<uint32_t>(j / kAcc) & 1u, abort_flag)) { ok = false; break; }
            if (!wait_bar(B.sc_full(ab), static_cast<uint32_t>(j / kAcc) & 1u, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const float *sw = scales + ab * 256;
            const float *sa = sw + 128 + 64 * hcol;
            const float dw = sw[r];
            const float2 dw2 = make_float2(dw, dw);
            const uint32_t taddr =
                tmem + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(ab * BN + 64 * hcol);
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                float p[32];
                tc_ld32(taddr + 32 * cc, p);
                if (cc == 1) {
                    tc_fence_before();
                    arrive(B.acc_empty(ab));  // TMEM buffer free for the next MMA
                }
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(sa + 32 * cc + i);
                    const float2 s01 = __fmul2_rn(dw2, make_float2(a4.x, a4.y));
                    const float2 s23 = __fmul2_rn(dw2, make_float2(a4.z, a4.w));
                    acc[16 * cc + i / 2] = __ffma2_rn(s01, make_float2(p[i], p[i + 1]), acc[16 * cc + i / 2]);
                    acc[16 * cc + i / 2 + 1] = __ffma2_rn(s23, make_float2(p[i + 2], p[i + 3]), acc[16 * cc + i / 2 + 1]);
                }
            }
            arrive(B.sc_empty(ab));
        }
        if (ok && !*abort_flag) {
            const int64_t row = n0 + r;
            if (row < n) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int64_t tok = t0 + 64 * hcol + 2 * i;
                    if (tok < t) y[tok * n + row] = acc[i].x;
                    if (tok + 1 < t) y[(tok + 1) * n + row] = acc[i].y;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

// ---------------------------------------------------------------------------
// host side: tensor maps through the driver entry point (no libcuda link)
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

bool make_map_2d(CUtensorMap *m, CUtensorMapDataType dt, int esize, const void *ptr, uint64_t d0, uint64_t d1,
                 uint64_t stride_bytes, uint32_t b0, uint32_t b1, CUtensorMapSwizzle sw)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {d0, d1};
    const cuuint64_t strides[1] = {stride_bytes};
    const cuuint32_t box[2] = {b0, b1};
    const cuuint32_t estr[2] = {1, 1};
    (void)esize;
    return fn(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

} // namespace

namespace q8 {

int gemm_take_error(cudaStream_t s)
{
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_gemm_err, sizeof(v), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_gemm_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return Q8_ERR_CUDA;
    return v ? Q8_ERR_DEVICE_TIMEOUT : Q8_OK;
}

// Requires k/32 % 8 == 0, 16-byte aligned pointers (checked by the caller).
int gemm_tc_launch(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, int64_t t, float *y,
                   cudaStream_t s)
{
    const int64_t nb = k / 32;
    const int64_t pitch = nb * 34;
    CUtensorMap ma, mb, md;
    if (!make_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, w, static_cast<uint64_t>(pitch / 2),
                     static_cast<uint64_t>(n), static_cast<uint64_t>(pitch), 136, BM, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, qs, static_cast<uint64_t>(k), static_cast<uint64_t>(t),
                     static_cast<uint64_t>(k), 128, BN, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&md, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, ds, static_cast<uint64_t>(nb), static_cast<uint64_t>(t),
                     static_cast<uint64_t>(nb * 4), 8, BN, CU_TENSOR_MAP_SWIZZLE_NONE))
        return Q8_ERR_LAUNCH;
    if (!set_max_dynamic_smem(reinterpret_cast<const void *>(gemm_tc_kernel), kSmemBytes, 2)) return Q8_ERR_LAUNCH;
    const dim3 grid(static_cast<unsigned>((n + BM - 1) / BM), static_cast<unsigned>((t + BN - 1) / BN));
    return launch_pdl(gemm_tc_kernel, grid, dim3(kThreads), kSmemBytes, s, ma, mb, md, n, t, static_cast<int>(nb), y);
}

} // namespace q8
