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
// Before the GEMM proper, a small pre-pass (gemm_prep_kernel) writes the
// plane's codes once per call into the caller's workspace as f16 tokens x k
// ("prepared operand"), so the GEMM loads them with TMA directly in the layout
// the tensor core reads -- every weight tile reuses it, instead of converting
// the same activation in every CTA.
//
// One CTA computes a 128 (weight rows) x 192 (tokens) tile over all of k.
// Per 32-wide block two K=16 MMAs produce the exact integer partial P in one
// of two TMEM buffers; the epilogue adds (d_w * d_a) * P to f32 register
// accumulators.  Every block needs a round trip between the tensor core and
// the epilogue (MMA completion -> epilogue -> buffer free), so tiles are wide
// (192 tokens); and a TMEM load takes ~130 cycles to land while
// tcgen05.wait::ld waits for all of a thread's loads, so the epilogue runs
// three warps per TMEM lane quarter (64 tokens and 64 accumulators each) to
// hide that latency.
// The tensor core queues little ahead of the thread issuing to it, so each
// TMEM buffer has its own issuing thread, and the epilogue is bound by its
// f32 work (one scale product and one fma per output and block).
// Warp roles (640 threads; setmaxnreg moves registers to the epilogue):
//   warp 0      TMA producer for raw Q8_0 weight rows (8 blocks per stage)
//   warp 1      TMEM allocator; MMA issuer (one thread) for the even blocks
//   warp 2      TMA producer for the prepared activation (2 blocks per stage)
//   warp 3      MMA issuer (one thread) for the odd blocks
//   warps 4-7   converters: one weight row each, raw int8 -> f16 canonical
//               K-major tile; the block's d_w (row) and d_a (256 tokens, read
//               from the plane) as f32 into a scale ring
//   warps 8-19  epilogue: three warps per TMEM lane quarter, 64 tokens each,
//               read in the 16x256b shape (4 rows x 16 tokens per thread and
//               load), packed f32x2 multiply/fma, 64 accumulators per thread
// Every mbarrier wait is bounded; a wait that runs out sets the CTA abort
// flag and the library error word, and all roles drain and exit.
#include <cuda.h>

#include <mutex>

#include "q8_common.cuh"

namespace {

__device__ unsigned int g_gemm_err;

constexpr int BM = 128, BN = 192;
constexpr int kABlocksPerStage = 8;                // raw weight stage: 8 blocks = 272 bytes per row
constexpr int kBBlocksPerStage = 2;                // prepared activation stage: 2 blocks = 64 f16 per token
constexpr int kAStages = 2, kBStages = 3, kF16Slots = 4, kScSlots = 4, kAcc = 2;
constexpr int kEpiCols = 64;                       // token columns per epilogue warp
constexpr int kEpiWarps = 4 * (BN / kEpiCols);     // 12: three per TMEM lane quarter
constexpr int kTmemBuf = 256;                      // column stride of the accumulator buffers
constexpr int kTmemCols = kAcc * kTmemBuf;         // 512 (allocations are powers of two)
static_assert(kBBlocksPerStage == kAcc, "each activation stage feeds one block of each MMA issuer");
constexpr int kConvThreads = 128;                  // warps 4-7
constexpr int kEpiThreads = 32 * kEpiWarps;        // 384: warps 8-19
constexpr int kThreads = 256 + kEpiThreads;        // 640
// registers per thread after setmaxnreg (launch: 96 x 640 = 61440 in the pool):
// 128*32 + 128*72 + 384*120 = 59392
constexpr int kRegsCtl = 32, kRegsConv = 72, kRegsEpi = 120;
static_assert(128 * kRegsCtl + 128 * kRegsConv + kEpiThreads * kRegsEpi <= 96 * kThreads, "register split");

constexpr int kARawBytes = BM * 272;               // 34816
constexpr int kBStageBytes = BN * 128;             // 24576: 192 tokens x 64 f16, 128B swizzle
constexpr int kA16Tile = BM * 64;                  // 8192: 128 rows x 32 f16, no swizzle
constexpr int kScBytes = (BM + BN) * 4;            // 1280: d_w[128], d_a[192] as f32

// shared-memory map (offsets from a 1024-byte aligned base)
constexpr int OFF_B = 0;                                        // 3 x 24576 (1024-aligned)
constexpr int OFF_ARAW = OFF_B + kBStages * kBStageBytes;       // 73728
constexpr int OFF_A16 = OFF_ARAW + kAStages * kARawBytes;       // 143360
constexpr int OFF_SC = OFF_A16 + kF16Slots * kA16Tile;          // 176128
constexpr int OFF_BAR = OFF_SC + kScSlots * kScBytes;           // 181248
static_assert(kBStageBytes % 1024 == 0 && OFF_A16 % 1024 == 0, "swizzle atoms and tiles stay aligned");
constexpr int kNumBars = 2 * kAStages + 2 * kBStages + 2 * kF16Slots + 2 * kScSlots + 2 * kAcc + kAcc;  // 32
constexpr int OFF_MISC = OFF_BAR + kNumBars * 8 + 8;
constexpr int kSmemBytes = OFF_MISC + 16 + 1024;                // + alignment slack

// ---------------------------------------------------------------------------
// PTX wrappers specific to this kernel
// ---------------------------------------------------------------------------
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

// 16 lanes x 32 columns (16x256b shape, 4 repetitions along the columns) ->
// 16 registers per thread.  Thread i of the warp receives, for repetition
// rep, lanes (i/4) and (i/4 + 8) of the 16 at columns 8*rep + 2*(i%4) + {0,1}:
// registers 4*rep + {0,1} (lane i/4), 4*rep + {2,3} (lane i/4 + 8).
// Asynchronous: the registers are valid only after tc_wait_ld16.
__device__ __forceinline__ void tc_ld16x256b_x4(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// Wait for this thread's outstanding TMEM loads.  The registers of the load
// being waited for pass through the statement, so no use of them can be
// scheduled before it; having no memory clobber, it leaves shared-memory
// loads free to move across it.
__device__ __forceinline__ void tc_wait_ld16(uint32_t (&r)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]));
}

// Shared-memory matrix descriptor, K-major.  No swizzle: core matrices of
// 8 rows x 16 bytes, LBO = byte step between core matrices along k, SBO =
// byte step between 8-row groups.  128-byte swizzle: rows of 128 bytes in
// 1024-byte atoms of 8 rows, SBO = 1024, LBO unused; a k offset inside the
// atom is added to the start address.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, bool sw128 = false)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((addr >> 4) & 0x3fffu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3fffu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3fffu) << 32;
    d |= static_cast<uint64_t>(1) << 46;  // descriptor version for tcgen05
    if (sw128) d |= static_cast<uint64_t>(2) << 61;
    return d;                             // base offset 0
}

// Instruction descriptor: D f32, A and B f16, both K-major, M = 128, N = BN.
constexpr uint32_t kIdesc = (1u << 4) | (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);

__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)  // no suspend-time hint: a suspended waiter wakes late
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

// Scale-ring order.  The epilogue reads TMEM in the 16x256b shape, so each
// of its threads holds four weight rows (32q + 16*sub + g + 8*e) and, per
// 32-column group cg of its 64 tokens, eight token columns
// (64h + 32cg + 8*rep + 2m + {0,1}); the converters store d_w and d_a so that
// those sets are contiguous, which makes the epilogue's scale reads 16-byte,
// bank-conflict-free loads.
__device__ __forceinline__ int dw_slot(int r)  // weight row 0..127
{
    return (r >> 5) * 32 + (r & 7) * 4 + ((r >> 4) & 1) * 2 + ((r >> 3) & 1);
}
__device__ __forceinline__ int da_slot(int c)  // token column 0..BN-1
{
    return (c >> 6) * 64 + ((c >> 5) & 1) * 32 + ((c >> 1) & 3) * 8 + ((c >> 3) & 3) * 2 + (c & 1);
}

// Converter step for weight row r, raw block BETA of the stage: read the 48
// bytes (three 16-byte aligned, bank-conflict-free loads) that contain the
// row's 34-byte block, write the 32 codes as f16 into the A tile and d_w as
// f32 into the scale ring (at dw_slot(r)).
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
    sw[dw_slot(r)] = __half2float(__ushort_as_half(static_cast<unsigned short>(dbits)));
    uint32_t qw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int ob = o + 2 + 4 * i;   // compile-time after unrolling
        qw[i] = (ob & 3) ? __byte_perm(w[ob >> 2], w[(ob >> 2) + 1], 0x5432) : w[ob >> 2];
    }
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) {
        uint4 v;
        q8::i8x4_to_f16x4(qw[2 * kc], v.x, v.y);
        q8::i8x4_to_f16x4(qw[2 * kc + 1], v.z, v.w);
        *reinterpret_cast<uint4 *>(a16 + (r >> 3) * 512 + kc * 128 + (r & 7) * 16) = v;
    }
}

// Epilogue step for one 16x256b.x4 load (two rows x eight token columns of
// this thread): acc += (d_w * d_a) * P in token pairs.  The scale d_w * d_a
// is rounded once before the fma, the order every block follows.
__device__ __forceinline__ void epi_math(float2 *acc, const uint32_t (&p)[16], const float (&da)[8], float dw_lo,
                                         float dw_hi)
{
    const float2 w0 = make_float2(dw_lo, dw_lo), w1 = make_float2(dw_hi, dw_hi);
#pragma unroll
    for (int rep = 0; rep < 4; ++rep) {
        const float2 d2 = make_float2(da[2 * rep], da[2 * rep + 1]);
        const float2 s0 = __fmul2_rn(w0, d2);
        const float2 s1 = __fmul2_rn(w1, d2);
        acc[2 * rep] = __ffma2_rn(s0, make_float2(__uint_as_float(p[4 * rep]), __uint_as_float(p[4 * rep + 1])),
                                  acc[2 * rep]);
        acc[2 * rep + 1] = __ffma2_rn(
            s1, make_float2(__uint_as_float(p[4 * rep + 2]), __uint_as_float(p[4 * rep + 3])), acc[2 * rep + 1]);
    }
}

struct Bars {
    uint32_t b0;
    __device__ uint32_t at(int i) const { return b0 + 8u * i; }
    __device__ uint32_t a_full(int s) const { return at(s); }
    __device__ uint32_t a_empty(int s) const { return at(kAStages + s); }
    __device__ uint32_t b_full(int s) const { return at(2 * kAStages + s); }
    __device__ uint32_t b_empty(int s) const { return at(2 * kAStages + kBStages + s); }
    __device__ uint32_t f_full(int s) const { return at(2 * kAStages + 2 * kBStages + s); }
    __device__ uint32_t f_empty(int s) const { return at(2 * kAStages + 2 * kBStages + kF16Slots + s); }
    __device__ uint32_t sc_full(int s) const { return at(2 * kAStages + 2 * kBStages + 2 * kF16Slots + s); }
    __device__ uint32_t sc_empty(int s) const
    {
        return at(2 * kAStages + 2 * kBStages + 2 * kF16Slots + kScSlots + s);
    }
    __device__ uint32_t acc_full(int s) const { return at(2 * kAStages + 2 * kBStages + 2 * kF16Slots + 2 * kScSlots + s); }
    __device__ uint32_t acc_empty(int s) const
    {
        return at(2 * kAStages + 2 * kBStages + 2 * kF16Slots + 2 * kScSlots + kAcc + s);
    }
    __device__ uint32_t drain(int issuer) const { return at(kNumBars - kAcc + issuer); }
};

// The d_a words of the 8 blocks of a raw weight stage for the tile's tokens
// r and r + 128 (32 contiguous bytes of the plane's ds row each); 0 for
// tokens past t, and the second one only exists for r + 128 < BN.
struct StageDa {
    uint32_t w[2][8];
};

__device__ __forceinline__ StageDa load_stage_da(const uint32_t *__restrict__ ds, int64_t nb, int64_t t, int64_t tok0,
                                                 int r, int s)
{
    StageDa d;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int64_t tok = tok0 + 128 * h;
        if (tok < t && (h == 0 || r + 128 < BN)) {
            const uint4 *p = reinterpret_cast<const uint4 *>(ds + tok * nb + 8 * s);
            const uint4 a = __ldg(p), b = __ldg(p + 1);
            d.w[h][0] = a.x; d.w[h][1] = a.y; d.w[h][2] = a.z; d.w[h][3] = a.w;
            d.w[h][4] = b.x; d.w[h][5] = b.y; d.w[h][6] = b.z; d.w[h][7] = b.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) d.w[h][i] = 0u;
        }
    }
    return d;
}

// One 32-wide block of a raw weight stage for the converter role.
template <int BETA>
__device__ __forceinline__ bool convert_block(const Bars &B, uint8_t *sm, int s, int r, const StageDa &da,
                                              volatile int *abort_flag)
{
    const int slot = s % kAStages;
    const int j = s * kABlocksPerStage + BETA;
    constexpr int fs = BETA % kF16Slots, ss = BETA % kScSlots;
    if (!wait_bar(B.f_empty(fs), (static_cast<uint32_t>(j / kF16Slots) & 1u) ^ 1u, abort_flag)) return false;
    if (!wait_bar(B.sc_empty(ss), (static_cast<uint32_t>(j / kScSlots) & 1u) ^ 1u, abort_flag)) return false;
    float *sw = reinterpret_cast<float *>(sm + OFF_SC + ss * kScBytes);
    float *sa = sw + BM;
    convert_a_row<BETA>(sm + OFF_ARAW + slot * kARawBytes + r * 272, sm + OFF_A16 + fs * kA16Tile, sw, r);
    sa[da_slot(r)] = __half2float(__ushort_as_half(static_cast<unsigned short>(da.w[0][BETA] & 0xffffu)));
    if (r + 128 < BN)
        sa[da_slot(r + 128)] = __half2float(__ushort_as_half(static_cast<unsigned short>(da.w[1][BETA] & 0xffffu)));
    q8::fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
    arrive(B.f_full(fs));
    arrive(B.sc_full(ss));
    if (BETA == kABlocksPerStage - 1) arrive(B.a_empty(slot));
    return true;
}

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }

__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const uint32_t *__restrict__ ds, int64_t n, int64_t t, int nb, float *__restrict__ y)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = q8::smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t *sm = smem_raw + (base - raw_base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Bars B{base + OFF_BAR};
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_MISC);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_MISC + 4);

    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * BM;
    const int64_t t0 = static_cast<int64_t>(blockIdx.y) * BN;

    if (threadIdx.x == 0) {
        *abort_flag = (*reinterpret_cast<volatile unsigned int *>(&g_gemm_err) != 0u) ? 1 : 0;
        uint64_t *b = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
        int i = 0;
        for (int k = 0; k < kAStages; ++k) q8::mbar_init(b + i++, 1);              // a_full: TMA bytes
        for (int k = 0; k < kAStages; ++k) q8::mbar_init(b + i++, kConvThreads);   // a_empty
        for (int k = 0; k < kBStages; ++k) q8::mbar_init(b + i++, 1);              // b_full: TMA bytes
        for (int k = 0; k < kBStages; ++k) q8::mbar_init(b + i++, kAcc);           // b_empty: one commit per issuer
        for (int k = 0; k < kF16Slots; ++k) q8::mbar_init(b + i++, kConvThreads);  // f_full
        for (int k = 0; k < kF16Slots; ++k) q8::mbar_init(b + i++, 1);             // f_empty: tcgen05.commit
        for (int k = 0; k < kScSlots; ++k) q8::mbar_init(b + i++, kConvThreads);   // sc_full
        for (int k = 0; k < kScSlots; ++k) q8::mbar_init(b + i++, kEpiThreads);    // sc_empty
        for (int k = 0; k < kAcc; ++k) q8::mbar_init(b + i++, 1);                  // acc_full: tcgen05.commit
        for (int k = 0; k < kAcc; ++k) q8::mbar_init(b + i++, kEpiThreads);        // acc_empty
        for (int k = 0; k < kAcc; ++k) q8::mbar_init(b + i++, 1);                  // MMA drain, per issuer
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
    if (warp < 4) {
        setmaxnreg_dec<kRegsCtl>();
        if (warp == 0 || warp == 2) {
            // -------------------------------------------------------- TMA producers
            if (lane == 0) {
                // Inputs may come from the previous kernel on the stream; the
                // converters also wait before reading the plane's scales, and Y
                // is written after the last MMA.
                q8::griddep_wait();
                const bool is_a = warp == 0;
                const int nstages = is_a ? nb / kABlocksPerStage : nb / kBBlocksPerStage;
                const int nbuf = is_a ? kAStages : kBStages;
                int issued = 0;
                for (int s = 0; s < nstages && !*abort_flag; ++s) {
                    const int slot = s % nbuf;
                    const uint32_t use = static_cast<uint32_t>(s / nbuf);
                    if (is_a) {
                        if (!wait_bar(B.a_empty(slot), (use & 1u) ^ 1u, abort_flag)) break;
                        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(B.a_full(slot)),
                                     "r"(kARawBytes)
                                     : "memory");
                        q8::tma_load_2d(base + OFF_ARAW + slot * kARawBytes, &tmA, s * 136, static_cast<int>(n0),
                                    B.a_full(slot));
                    } else {
                        if (!wait_bar(B.b_empty(slot), (use & 1u) ^ 1u, abort_flag)) break;
                        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(B.b_full(slot)),
                                     "r"(kBStageBytes)
                                     : "memory");
                        q8::tma_load_2d(base + OFF_B + slot * kBStageBytes, &tmB, s * 32 * kBBlocksPerStage,
                                    static_cast<int>(t0), B.b_full(slot));
                    }
                    issued = s + 1;
                }
                // drain: the last stages issued must have landed before the CTA exits
                for (int s = issued - nbuf < 0 ? 0 : issued - nbuf; s < issued; ++s)
                    drain_bar(is_a ? B.a_full(s % nbuf) : B.b_full(s % nbuf), static_cast<uint32_t>(s / nbuf) & 1u);
            }
        } else {
            // -------------------------------------------------------- MMA issuers
            // Warp 1 issues the even blocks (TMEM buffer 0), warp 3 the odd
            // ones (buffer 1).  The tensor core hardly queues ahead of the
            // issuing thread, so one issuer's barrier waits and bookkeeping
            // would stall the pipe between blocks; two issuers hide each
            // other's.
            const int who = warp == 1 ? 0 : 1;
            if (lane == 0) {
                for (int j = who; j < nb; j += kAcc) {
                    const int fs = j % kF16Slots, ab = who;
                    const int sb = (j / kBBlocksPerStage) % kBStages, bq = j % kBBlocksPerStage;
                    if (!wait_bar(B.f_full(fs), static_cast<uint32_t>(j / kF16Slots) & 1u, abort_flag)) break;
                    if (!wait_bar(B.b_full(sb), static_cast<uint32_t>(j / (kBBlocksPerStage * kBStages)) & 1u,
                                  abort_flag))
                        break;
                    if (!wait_bar(B.acc_empty(ab), (static_cast<uint32_t>(j / kAcc) & 1u) ^ 1u, abort_flag)) break;
                    tc_fence_after();
                    const uint32_t d = tmem + static_cast<uint32_t>(ab * kTmemBuf);
                    const uint32_t a_addr = base + OFF_A16 + fs * kA16Tile;
                    const uint32_t b_addr = base + OFF_B + sb * kBStageBytes + 64 * bq;
#pragma unroll
                    for (int kk = 0; kk < 2; ++kk)  // two K=16 steps = one 32-wide block
                        tc_mma_f16(d, smem_desc(a_addr + 256 * kk, 128, 512),
                                   smem_desc(b_addr + 32 * kk, 16, 1024, true), kIdesc, kk);
                    tc_commit(B.f_empty(fs));
                    tc_commit(B.acc_full(ab));
                    tc_commit(B.b_empty(sb));  // counts one commit from each issuer per stage
                }
                // drain: every MMA this thread issued must have completed before TMEM is freed
                tc_commit(B.drain(who));
                drain_bar(B.drain(who), 0);
            }
        }
    } else if (warp < 8) {
        setmaxnreg_dec<kRegsConv>();
        // ------------------------------------------------------------ converters
        const int r = threadIdx.x - 128;  // weight row of the tile and tokens r, r + 128 (if < BN), 0..127
        const int nstages = nb / kABlocksPerStage;
        q8::griddep_wait();               // the plane's scales may come from the previous kernel
        for (int s = 0; s < nstages && !*abort_flag; ++s) {
            const StageDa da = load_stage_da(ds, nb, t, t0 + r, r, s);
            if (!wait_bar(B.a_full(s % kAStages), static_cast<uint32_t>(s / kAStages) & 1u, abort_flag)) break;
            if (!convert_block<0>(B, sm, s, r, da, abort_flag)) break;
            if (!convert_block<1>(B, sm, s, r, da, abort_flag)) break;
            if (!convert_block<2>(B, sm, s, r, da, abort_flag)) break;
            if (!convert_block<3>(B, sm, s, r, da, abort_flag)) break;
            if (!convert_block<4>(B, sm, s, r, da, abort_flag)) break;
            if (!convert_block<5>(B, sm, s, r, da, abort_flag)) break;
            if (!convert_block<6>(B, sm, s, r, da, abort_flag)) break;
            if (!convert_block<7>(B, sm, s, r, da, abort_flag)) break;
        }
    } else {
        setmaxnreg_inc<kRegsEpi>();
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;            // TMEM lane quarter of this warp
        const int hcol = (warp - 8) >> 2;  // token group: [64*hcol, 64*hcol + 64)
        const int g = lane >> 2, m = lane & 3;
        // this thread's outputs: rows 32q + 16*sub + g + 8*e, token columns
        // 64*hcol + 32*cg + 8*rep + 2m + {0,1}; acc index 8*(2cg + sub) + 2*rep + e
        float2 acc[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = make_float2(0.0f, 0.0f);
        bool ok = true;
        for (int j = 0; j < nb; ++j) {
            const int ab = j % kAcc, ss = j % kScSlots;
            if (!wait_bar(B.acc_full(ab), static_cast<uint32_t>(j / kAcc) & 1u, abort_flag)) { ok = false; break; }
            if (!wait_bar(B.sc_full(ss), static_cast<uint32_t>(j / kScSlots) & 1u, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const float *sw = reinterpret_cast<const float *>(sm + OFF_SC + ss * kScBytes);
            const float4 w4 = *reinterpret_cast<const float4 *>(sw + 32 * q + 4 * g);  // dw_slot order
            const float *sa = sw + BM + kEpiCols * hcol + 8 * m;                        // da_slot order, + 32*cg
            const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) +
                                   static_cast<uint32_t>(ab * kTmemBuf + kEpiCols * hcol);
            // chunk c = (cg = c / 2, sub = c % 2): 16 lanes x 32 columns.  Loads
            // are double-buffered: chunk c + 1 is in flight while chunk c is
            // scaled and accumulated.  The buffer is released once its last
            // chunk is in registers.
            uint32_t p0[16], p1[16];
            float da[8];
            tc_ld16x256b_x4(tbase, p0);
            tc_wait_ld16(p0);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t(&cur)[16] = (c & 1) ? p1 : p0;
                uint32_t(&nxt)[16] = (c & 1) ? p0 : p1;
                if ((c & 1) == 0) {
                    const float4 a0 = *reinterpret_cast<const float4 *>(sa + 32 * (c >> 1));
                    const float4 a1 = *reinterpret_cast<const float4 *>(sa + 32 * (c >> 1) + 4);
                    da[0] = a0.x; da[1] = a0.y; da[2] = a0.z; da[3] = a0.w;
                    da[4] = a1.x; da[5] = a1.y; da[6] = a1.z; da[7] = a1.w;
                }
                if (c < 3) {
                    const int cn = c + 1;
                    tc_ld16x256b_x4(tbase + (static_cast<uint32_t>(16 * (cn & 1)) << 16) + 32 * (cn >> 1), nxt);
                }
                if (c & 1) epi_math(acc + 8 * c, cur, da, w4.z, w4.w);
                else epi_math(acc + 8 * c, cur, da, w4.x, w4.y);
                if (c < 3) tc_wait_ld16(nxt);
                if (c == 2) {
                    tc_fence_before();
                    arrive(B.acc_empty(ab));  // TMEM buffer free for the next block's MMAs
                }
            }
            arrive(B.sc_empty(ss));
        }
        if (ok && !*abort_flag) {
#pragma unroll
            for (int c = 0; c < 4; ++c) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int64_t row = n0 + 32 * q + 16 * (c & 1) + g + 8 * e;
                    if (row >= n) continue;
#pragma unroll
                    for (int rep = 0; rep < 4; ++rep) {
                        const int64_t tok = t0 + kEpiCols * hcol + 32 * (c >> 1) + 8 * rep + 2 * m;
                        const float2 v = acc[8 * c + 2 * rep + e];
                        if (tok < t) y[tok * n + row] = v.x;
                        if (tok + 1 < t) y[(tok + 1) * n + row] = v.y;
                    }
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

// Pre-pass: plane codes (qs) rows [0, t) -> prepared operand b16[t][k] = f16(q), exact.
__global__ void __launch_bounds__(256)
gemm_prep_kernel(const uint4 *__restrict__ qs, int64_t t, int64_t k, uint4 *__restrict__ b16)
{
    q8::griddep_launch_dependents();
    q8::griddep_wait();  // the plane may come from the previous kernel
    const int64_t total = t * (k / 16);  // 16-code chunks; qs row stride k: flat index
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint4 v = __ldg(qs + i);
        uint4 o0, o1;
        q8::i8x4_to_f16x4(v.x, o0.x, o0.y);
        q8::i8x4_to_f16x4(v.y, o0.z, o0.w);
        q8::i8x4_to_f16x4(v.z, o1.x, o1.y);
        q8::i8x4_to_f16x4(v.w, o1.z, o1.w);
        b16[2 * i] = o0;
        b16[2 * i + 1] = o1;
    }
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

size_t gemm_workspace_bytes(int64_t t, int64_t k)
{
    return static_cast<size_t>(t) * static_cast<size_t>(k) * 2;  // the prepared f16 codes
}

// Requires k/32 % 8 == 0, 16-byte aligned pointers and a workspace of at least
// gemm_workspace_bytes(t, k) bytes (checked by the caller).
int gemm_tc_launch(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, int64_t t, float *y,
                   void *workspace, cudaStream_t s)
{
    const int64_t nb = k / 32;
    const int64_t pitch = nb * 34;
    uint8_t *b16 = static_cast<uint8_t *>(workspace);
    CUtensorMap ma, mb;
    if (!make_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT16, w, static_cast<uint64_t>(pitch / 2),
                     static_cast<uint64_t>(n), static_cast<uint64_t>(pitch), 136, BM, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT16, b16, static_cast<uint64_t>(k), static_cast<uint64_t>(t),
                     static_cast<uint64_t>(k * 2), 64, BN, CU_TENSOR_MAP_SWIZZLE_128B))
        return Q8_ERR_LAUNCH;
    const int sms = device_sm_count();
    const int64_t chunks = t * (k / 16);
    int64_t pgrid = (chunks + 255) / 256;
    const int64_t pcap = static_cast<int64_t>(sms > 0 ? sms : 152) * 8;
    pgrid = pgrid < pcap ? pgrid : pcap;
    int st = launch_pdl(gemm_prep_kernel, dim3(static_cast<unsigned>(pgrid)), dim3(256), 0, s,
                        reinterpret_cast<const uint4 *>(qs), t, k, reinterpret_cast<uint4 *>(b16));
    if (st != Q8_OK) return st;
    if (!set_max_dynamic_smem(reinterpret_cast<const void *>(gemm_tc_kernel), kSmemBytes, 2)) return Q8_ERR_LAUNCH;
    const dim3 grid(static_cast<unsigned>((n + BM - 1) / BM), static_cast<unsigned>((t + BN - 1) / BN));
    return launch_pdl(gemm_tc_kernel, grid, dim3(kThreads), kSmemBytes, s, ma, mb, ds, n, t, static_cast<int>(nb), y);
}

} // namespace q8

// ---------------------------------------------------------------------------
// q8_0_gemm_noalloc: the same GEMM with its scratch in a fixed device array.
//
// Some callers cannot allocate device memory on the way to this call: a
// serving engine that reserved all of the GPU's memory for its own pool at
// start-up, a plugin whose host forbids allocation once it is initialised,
// or a latency-critical path that cannot afford cudaMalloc's implicit
// synchronisation.  For them the prepared activation lives in the array
// below.  It is part of the library's device image, so every GPU on which
// this library's GEMM module is loaded keeps these bytes until the process
// exits, whether or not this entry point is ever called.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(32) << 20;  // 32 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64];  // device address of g_noalloc_scratch, per device ordinal

// Device address of the scratch array on the current device, looked up once
// per device (the array's name in host code is only a stand-in for it).
int noalloc_scratch(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return Q8_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return Q8_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return Q8_OK;
}

} // namespace

extern "C" int q8_0_gemm_noalloc(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds,
                                 int64_t t, int64_t rows_pad, float *y, void *stream)
{
    if (!w || !qs || !ds || !y || n < 1 || t < 1 || k <= 0 || (k % 32) != 0 || rows_pad < t) return Q8_ERR_ARG;
    const size_t need = q8_0_gemm_workspace_bytes(t, k);
    if (need > kNoAllocScratchBytes) return Q8_ERR_TOO_BIG;
    if (!q8::aligned16(w) || !q8::aligned16(qs) || !q8::aligned16(ds) || !q8::aligned16(y)) return Q8_ERR_ALIGN;
    if (!q8::device_is_sm103()) return Q8_ERR_DEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (t == 1) return q8_0_gemv(w, n, k, qs, ds, y, stream);  // these shapes need no scratch
    if ((k / 32) % 8 != 0) {
        if (t > 65535) return Q8_ERR_ARG;
        return q8::gemv_generic_launch(w, n, k, qs, ds, y, t, s);
    }
    if (t <= Q8_GEMV_MAX_TOKENS) return q8::gemv_small_launch(w, n, k, qs, ds, y, t, s);
    if (t > int64_t(65535) * 128 || n > (int64_t(1) << 31) - 128) return Q8_ERR_ARG;
    void *scratch = nullptr;
    const int st = noalloc_scratch(&scratch);
    if (st != Q8_OK) return st;
    return q8::gemm_tc_launch(w, n, k, qs, ds, t, y, scratch, s);
}

extern "C" size_t q8_0_gemm_noalloc_max_bytes(void) { return kNoAllocScratchBytes; }

