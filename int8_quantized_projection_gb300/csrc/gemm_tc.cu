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
// structural rewrite spec" (sec. 2) and the q8_0 plane of "54 - r51 -
// producer-fused A-quantize mode 1" (sec. 2.1).
//
// Two pre-passes write the operands once per call into the caller's
// workspace in the form the tensor core and the epilogue read: the weight
// codes as f16 [n][k] with each block's d_w as f32, and the plane's codes as
// f16 [t][k] with each block's d_a as f32; the scales are stored per
// (tile, block) in the order the epilogue threads read them.  The GEMM then
// only moves data with TMA -- the weight codes are widened once per call, not
// once per token tile -- and its warps are MMA issuers and epilogue.
//
// One CTA computes a 128 (weight rows) x 192 (tokens) tile over all of k.
// Per 32-wide block two K=16 MMAs produce the exact integer partial P in one
// of two TMEM buffers; the epilogue adds (d_w * d_a) * P to f32 register
// accumulators.  Every block needs a round trip between the tensor core and
// the epilogue (MMA completion -> epilogue -> buffer free).  The tensor core
// queues little ahead of the thread issuing to it, so each TMEM buffer has
// its own issuing thread.  A TMEM load takes ~130 cycles to land and
// tcgen05.wait::ld waits for all of a thread's loads, so each epilogue thread
// reads its share of a block (64 values) in two halves: the first half's
// loads and wait, then the second half's loads in flight while the first
// half is scaled and accumulated, then the buffer is freed and the second
// half's math follows; three warps per TMEM lane quarter keep the f32 pipe
// busy meanwhile.
// Warp roles (512 threads; setmaxnreg moves registers to the epilogue):
//   warp 0      TMA producer: the weight and activation tiles of 2 blocks
//   warp 1      TMEM allocator; MMA issuer (one thread) for the even blocks
//   warp 2      bulk-copy producer: the d_w and d_a of 4 blocks per ring slot
//   warp 3      MMA issuer (one thread) for the odd blocks
//   warps 4-15  epilogue: three warps per TMEM lane quarter, 64 tokens each,
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
constexpr int kStageBlocks = 2;                    // 32-wide blocks per operand stage (128 bytes of f16 per row)
constexpr int kStages = 4, kScSlots = 4, kAcc = 2;
static_assert(kStageBlocks == kAcc, "each stage feeds one block of each MMA issuer");
constexpr int kEpiCols = 64;                       // token columns per epilogue warp
constexpr int kEpiWarps = 4 * (BN / kEpiCols);     // 12: three per TMEM lane quarter
constexpr int kTmemBuf = 256;                      // column stride of the accumulator buffers
constexpr int kTmemCols = kAcc * kTmemBuf;         // 512 (allocations are powers of two)
constexpr int kEpiThreads = 32 * kEpiWarps;        // 384: warps 4-15
constexpr int kThreads = 128 + kEpiThreads;        // 512
// registers per thread after setmaxnreg (launch: 128 x 512 = 65536 in the pool)
constexpr int kRegsCtl = 32, kRegsEpi = 160;
static_assert(128 * kRegsCtl + kEpiThreads * kRegsEpi <= 128 * kThreads, "register split");

constexpr int kATileBytes = BM * 128;              // 16384: 128 rows x 64 f16, 128B swizzle
constexpr int kBTileBytes = BN * 128;              // 24576: 192 tokens x 64 f16, 128B swizzle
constexpr int kStageBytes = kATileBytes + kBTileBytes;  // 40960
constexpr int kScBytes = (BM + BN) * 4;            // 1280: d_w[128], d_a[192] as f32, per block
#ifndef Q8_GEMM_SC_GROUP
#define Q8_GEMM_SC_GROUP 4
#endif
constexpr int kScGroup = Q8_GEMM_SC_GROUP;         // blocks whose scales share a ring slot (one wait per group)
constexpr int kScSlotBytes = kScGroup * kScBytes;  // 5120: d_w[4][128], then d_a[4][192]
static_assert(kScGroup >= 1 && kScGroup <= 8, "scale slots fit beside the operand stages");

// shared-memory map (offsets from a 1024-byte aligned base)
constexpr int OFF_STAGE = 0;                                    // 4 x 40960
constexpr int OFF_SC = OFF_STAGE + kStages * kStageBytes;       // 163840
constexpr int OFF_BAR = OFF_SC + kScSlots * kScSlotBytes;       // 184320 (kScGroup = 4)
static_assert(kStageBytes % 1024 == 0 && kATileBytes % 1024 == 0, "swizzle atoms stay aligned");
constexpr int kNumBars = 2 * kStages + 2 * kScSlots + 2 * kAcc + kAcc;  // 22
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
// Asynchronous: the registers are valid only after tc_wait_ld_all, and
// tc_regs16 keeps their uses from being scheduled before that wait.
__device__ __forceinline__ void tc_ld16x256b_x4(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
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

// Wait for this thread's outstanding TMEM loads, without naming registers
// (pair with tc_regs16 on every register those loads filled).
__device__ __forceinline__ void tc_wait_ld_all() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Pass 16 registers through an empty statement placed after the wait, so no
// use of them can be scheduled before it.
__device__ __forceinline__ void tc_regs16(uint32_t (&r)[16])
{
    asm volatile(""
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]));
}

// Pass 16 accumulator pairs through an empty statement: the arithmetic that
// produced them is done before any later volatile statement (a TMEM wait).
__device__ __forceinline__ void acc_order16(float2 *a)
{
    asm volatile(""
                 : "+f"(a[0].x), "+f"(a[0].y), "+f"(a[1].x), "+f"(a[1].y), "+f"(a[2].x), "+f"(a[2].y), "+f"(a[3].x),
                   "+f"(a[3].y), "+f"(a[4].x), "+f"(a[4].y), "+f"(a[5].x), "+f"(a[5].y), "+f"(a[6].x), "+f"(a[6].y),
                   "+f"(a[7].x), "+f"(a[7].y), "+f"(a[8].x), "+f"(a[8].y), "+f"(a[9].x), "+f"(a[9].y), "+f"(a[10].x),
                   "+f"(a[10].y), "+f"(a[11].x), "+f"(a[11].y), "+f"(a[12].x), "+f"(a[12].y), "+f"(a[13].x),
                   "+f"(a[13].y), "+f"(a[14].x), "+f"(a[14].y), "+f"(a[15].x), "+f"(a[15].y));
}

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
    if (Q8_WAIT_LIMIT_NS == 0) {  // a build that gives up at once: one non-blocking test
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok) return true;
        *abort_flag = 1;
        atomicOr(&g_gemm_err, 1u);
        return false;
    }
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
        if (q8::globaltimer_ns() - t0 > Q8_DRAIN_LIMIT_NS) {
            atomicOr(&g_gemm_err, 1u);
            return;
        }
    }
}

__device__ __forceinline__ void arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Scale order.  The epilogue reads TMEM in the 16x256b shape, so each of its
// threads holds four weight rows (32q + 16*sub + g + 8*e) and, per 32-column
// group cg of its 64 tokens, eight token columns (64h + 32cg + 8*rep + 2m +
// {0,1}); the pre-passes store d_w and d_a so that those sets are contiguous,
// which makes the epilogue's scale reads 16-byte, bank-conflict-free loads.
__device__ __forceinline__ int dw_slot(int r)  // weight row 0..127
{
    return (r >> 5) * 32 + (r & 7) * 4 + ((r >> 4) & 1) * 2 + ((r >> 3) & 1);
}
// (da_slot is the definition of the order; the activation pre-pass writes
// its inverse, and the epilogue reads slots in this order.)
__device__ __forceinline__ __attribute__((unused)) int da_slot(int c)  // token column 0..BN-1
{
    return (c >> 6) * 64 + ((c >> 5) & 1) * 32 + ((c >> 1) & 3) * 8 + ((c >> 3) & 3) * 2 + (c & 1);
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
    __device__ uint32_t full(int s) const { return at(s); }                        // stage landed (TMA bytes)
    __device__ uint32_t empty(int s) const { return at(kStages + s); }             // both issuers' MMAs done
    __device__ uint32_t sc_full(int s) const { return at(2 * kStages + s); }       // scales landed
    __device__ uint32_t sc_empty(int s) const { return at(2 * kStages + kScSlots + s); }  // epilogue done
    __device__ uint32_t acc_full(int s) const { return at(2 * kStages + 2 * kScSlots + s); }
    __device__ uint32_t acc_empty(int s) const { return at(2 * kStages + 2 * kScSlots + kAcc + s); }
    __device__ uint32_t drain(int issuer) const { return at(kNumBars - kAcc + issuer); }
};

template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }

template <bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const float *__restrict__ dwt, const float *__restrict__ dat, int64_t n, int64_t t, int nb,
               float *__restrict__ y, float *__restrict__ part)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = q8::smem_u32(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t *sm = smem_raw + (base - raw_base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Bars B{base + OFF_BAR};
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + OFF_MISC);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + OFF_MISC + 4);

    // token tiles vary fastest, so the CTAs running together share weight rows in L2
    const int64_t n0 = static_cast<int64_t>(blockIdx.y) * BM;
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * BN;
    // split-K (gridDim.z > 1): this CTA takes stages [s0, s0 + nsl) of k and
    // writes its partial tile to part[z]; j below counts this CTA's blocks
    // (a separate instantiation, so the unsplit kernel carries none of it)
    const int nst = nb / kStageBlocks;
    const int s0 = kSplit ? static_cast<int>(static_cast<int64_t>(nst) * blockIdx.z / gridDim.z) : 0;
    const int nsl = kSplit ? static_cast<int>(static_cast<int64_t>(nst) * (blockIdx.z + 1) / gridDim.z) - s0 : nst;
    const int j0 = s0 * kStageBlocks, nbl = kSplit ? nsl * kStageBlocks : nb;
    float *out = kSplit ? part + static_cast<int64_t>(blockIdx.z) * t * n : y;

    if (threadIdx.x == 0) {
        *abort_flag = (*reinterpret_cast<volatile unsigned int *>(&g_gemm_err) != 0u) ? 1 : 0;
        uint64_t *b = reinterpret_cast<uint64_t *>(sm + OFF_BAR);
        int i = 0;
        for (int k = 0; k < kStages; ++k) q8::mbar_init(b + i++, 1);             // full: TMA bytes
        for (int k = 0; k < kStages; ++k) q8::mbar_init(b + i++, kAcc);          // empty: one commit per issuer
        for (int k = 0; k < kScSlots; ++k) q8::mbar_init(b + i++, 1);            // sc_full: copy bytes
        for (int k = 0; k < kScSlots; ++k) q8::mbar_init(b + i++, kEpiThreads);  // sc_empty
        for (int k = 0; k < kAcc; ++k) q8::mbar_init(b + i++, 1);                // acc_full: tcgen05.commit
        for (int k = 0; k < kAcc; ++k) q8::mbar_init(b + i++, kEpiThreads);      // acc_empty
        for (int k = 0; k < kAcc; ++k) q8::mbar_init(b + i++, 1);                // MMA drain, per issuer
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
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------------ operand producer
            // Inputs come from the pre-passes just before on the stream; Y is
            // written only after the last MMA, which follows these loads.
            q8::griddep_wait();
            int issued = 0;
            for (int s = 0; s < nsl && !*abort_flag; ++s) {
                const int slot = s % kStages;
                if (!wait_bar(B.empty(slot), (static_cast<uint32_t>(s / kStages) & 1u) ^ 1u, abort_flag)) break;
                q8::mbar_arrive_expect_tx(reinterpret_cast<uint64_t *>(sm + OFF_BAR) + slot, kStageBytes);
                const uint32_t dst = base + OFF_STAGE + slot * kStageBytes;
                const int kx = (s0 + s) * 32 * kStageBlocks;
                q8::tma_load_2d(dst, &tmA, kx, static_cast<int>(n0), B.full(slot));
                q8::tma_load_2d(dst + kATileBytes, &tmB, kx, static_cast<int>(t0), B.full(slot));
                issued = s + 1;
            }
            // drain: the last stages issued must have landed before the CTA exits
            for (int s = issued - kStages < 0 ? 0 : issued - kStages; s < issued; ++s)
                drain_bar(B.full(s % kStages), static_cast<uint32_t>(s / kStages) & 1u);
        } else if (warp == 2 && lane == 0) {
            // ------------------------------------------------------------ scale producer
            q8::griddep_wait();
            const float *dw_tile = dwt + (static_cast<int64_t>(blockIdx.y) * nb + j0) * BM;
            const float *da_tile = dat + (static_cast<int64_t>(blockIdx.x) * nb + j0) * BN;
            // one slot per group of kScGroup blocks (the last group may be short)
            const int ngr = (nbl + kScGroup - 1) / kScGroup;
            int issued = 0;
            for (int G = 0; G < ngr && !*abort_flag; ++G) {
                const int ss = G % kScSlots;
                if (!wait_bar(B.sc_empty(ss), (static_cast<uint32_t>(G / kScSlots) & 1u) ^ 1u, abort_flag)) break;
                const int nbk = nbl - G * kScGroup < kScGroup ? nbl - G * kScGroup : kScGroup;
                uint64_t *bar = reinterpret_cast<uint64_t *>(sm + OFF_BAR) + 2 * kStages + ss;
                q8::mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nbk * kScBytes));
                uint8_t *dst = sm + OFF_SC + ss * kScSlotBytes;
                q8::bulk_g2s(dst, dw_tile + static_cast<int64_t>(G) * kScGroup * BM, nbk * BM * 4, bar);
                q8::bulk_g2s(dst + kScGroup * BM * 4, da_tile + static_cast<int64_t>(G) * kScGroup * BN, nbk * BN * 4,
                             bar);
                issued = G + 1;
            }
            for (int G = issued - kScSlots < 0 ? 0 : issued - kScSlots; G < issued; ++G)
                drain_bar(B.sc_full(G % kScSlots), static_cast<uint32_t>(G / kScSlots) & 1u);
        } else if ((warp == 1 || warp == 3) && lane == 0) {
            // ------------------------------------------------------------ MMA issuers
            // Warp 1 issues the even blocks (TMEM buffer 0), warp 3 the odd
            // ones (buffer 1).
            const int who = warp == 1 ? 0 : 1;
            for (int j = who; j < nbl; j += kAcc) {
                const int st = (j / kStageBlocks) % kStages, bq = j % kStageBlocks;
                const uint32_t use = static_cast<uint32_t>(j / (kStageBlocks * kStages));
                if (!wait_bar(B.full(st), use & 1u, abort_flag)) break;
                if (!wait_bar(B.acc_empty(who), (static_cast<uint32_t>(j / kAcc) & 1u) ^ 1u, abort_flag)) break;
                tc_fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(who * kTmemBuf);
                const uint32_t a_addr = base + OFF_STAGE + st * kStageBytes + 64 * bq;
                const uint32_t b_addr = a_addr + kATileBytes;
#pragma unroll
                for (int kk = 0; kk < 2; ++kk)  // two K=16 steps = one 32-wide block
                    tc_mma_f16(d, smem_desc(a_addr + 32 * kk, 16, 1024, true),
                               smem_desc(b_addr + 32 * kk, 16, 1024, true), kIdesc, kk);
                tc_commit(B.empty(st));  // counts one commit from each issuer per stage
                tc_commit(B.acc_full(who));
            }
            // drain: every MMA this thread issued must have completed before TMEM is freed
            tc_commit(B.drain(who));
            drain_bar(B.drain(who), 0);
        }
    } else {
        setmaxnreg_inc<kRegsEpi>();
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;            // TMEM lane quarter of this warp
        const int hcol = (warp - 4) >> 2;  // token group: [64*hcol, 64*hcol + 64)
        const int g = lane >> 2, m = lane & 3;
        // this thread's outputs: rows 32q + 16*sub + g + 8*e, token columns
        // 64*hcol + 32*cg + 8*rep + 2m + {0,1}; acc index 8*(2cg + sub) + 2*rep + e
        float2 acc[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = make_float2(0.0f, 0.0f);
        bool ok = true;
        for (int j = 0; j < nbl; ++j) {
            const int ab = j % kAcc, grp = j / kScGroup, bq = j % kScGroup, ss = grp % kScSlots;
            if (!wait_bar(B.acc_full(ab), static_cast<uint32_t>(j / kAcc) & 1u, abort_flag)) { ok = false; break; }
            tc_fence_after();
            // the scale slot of this block's group: waited for at the group's first block
            if (bq == 0 &&
                !wait_bar(B.sc_full(ss), static_cast<uint32_t>(grp / kScSlots) & 1u, abort_flag)) {
                ok = false;
                break;
            }
            // the block's share in two halves of 32 token columns: chunk c =
            // (cg = c / 2, sub = c % 2) is 16 lanes x 32 columns.  The second
            // half's TMEM loads are in flight while the first half's math
            // runs; once they land the buffer is free for the MMAs of block j + 2
            const uint32_t tbase = tmem + (static_cast<uint32_t>(32 * q) << 16) +
                                   static_cast<uint32_t>(ab * kTmemBuf + kEpiCols * hcol);
            uint32_t p[4][16];
            tc_ld16x256b_x4(tbase, p[0]);
            tc_ld16x256b_x4(tbase + (16u << 16), p[1]);
            tc_wait_ld_all();
            tc_regs16(p[0]);
            tc_regs16(p[1]);
            tc_ld16x256b_x4(tbase + 32, p[2]);
            tc_ld16x256b_x4(tbase + (16u << 16) + 32, p[3]);
            const float *sw = reinterpret_cast<const float *>(sm + OFF_SC + ss * kScSlotBytes);
            const float4 w4 = *reinterpret_cast<const float4 *>(sw + bq * BM + 32 * q + 4 * g);  // dw_slot order
            const float *sa = sw + kScGroup * BM + bq * BN + kEpiCols * hcol + 8 * m;            // da_slot order, + 32*cg
            {
                const float4 a0 = *reinterpret_cast<const float4 *>(sa);
                const float4 a1 = *reinterpret_cast<const float4 *>(sa + 4);
                const float da[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                epi_math(acc, p[0], da, w4.x, w4.y);
                epi_math(acc + 8, p[1], da, w4.z, w4.w);
            }
            acc_order16(acc);  // the first half's math stays ahead of the second wait
            tc_wait_ld_all();
            tc_regs16(p[2]);
            tc_regs16(p[3]);
            tc_fence_before();
            arrive(B.acc_empty(ab));
            {
                const float4 a0 = *reinterpret_cast<const float4 *>(sa + 32);
                const float4 a1 = *reinterpret_cast<const float4 *>(sa + 36);
                const float da[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                epi_math(acc + 16, p[2], da, w4.x, w4.y);
                epi_math(acc + 24, p[3], da, w4.z, w4.w);
            }
            if (bq == kScGroup - 1 || j == nbl - 1) arrive(B.sc_empty(ss));  // the group's last block
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
                        if (tok < t) out[tok * n + row] = v.x;
                        if (tok + 1 < t) out[(tok + 1) * n + row] = v.y;
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

// Pre-pass over the weights: codes -> f16 [n][k] (exact) and each block's d_w
// as f32 into dwt[row tile][block][dw_slot(row % 128)] (0 for rows past n).
// A CTA takes one 32-row group of a tile and B consecutive blocks (B * 34
// bytes of each row, 16-byte aligned because k/32 % 8 == 0 and B % 8 == 0):
// each warp loads four row pieces with coalesced 16-byte loads (all in
// flight at once) to shared memory, then widens their (row, block) pairs,
// one per lane at a time, each writing its 64 bytes of f16.  The group's d_w slots are
// contiguous (32 per block), so the scales go through shared memory and out
// as one 128-byte store per block.  B = 32 when the items fill the GPU
// several times over; B = 8 spreads a small matrix over more SMs.
template <int B, int NT>
__global__ void __launch_bounds__(NT)
gemm_prep_w_kernel(const uint8_t *__restrict__ w, int64_t n, int nb, uint4 *__restrict__ a16, float *__restrict__ dwt)
{
    static_assert(B % 8 == 0 && B <= 32, "row pieces must be whole 16-byte words");
    constexpr int kWarps = NT / 32;
    constexpr int kRows = 32 / kWarps;                      // rows a warp loads and widens
    constexpr int kRowWords = B * 34 / 16;                  // 16-byte words per row piece
    constexpr int kWords = (kRowWords + 31) / 32;           // per lane and row
    constexpr int kPairs = kRows * B / 32;                  // (row, block) pairs per lane
    static_assert(kWarps * kRows == 32 && kPairs * 32 == kRows * B, "one 32-row group per CTA");
    __shared__ __align__(16) uint4 buf[32][kRowWords];
    __shared__ float sdw[B][33];  // [block][slot in the group], padded: conflict-free both ways
    q8::griddep_launch_dependents();
    q8::griddep_wait();  // the previous call may still read this workspace
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tiles = (n + BM - 1) / BM;
    const int chunks = (nb + B - 1) / B;  // per row
    const int64_t items = tiles * (BM / 32) * chunks;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int64_t grp = it / chunks;
        const int c = static_cast<int>(it - grp * chunks);
        const int64_t r0 = grp * 32;  // first row of the group
        const int b0 = c * B;
        const int cb = min(B, nb - b0);  // a multiple of 8
        const int n16 = cb * 34 / 16;
        uint4 v[kRows][kWords];
#pragma unroll
        for (int q = 0; q < kRows; ++q) {
            const int64_t r = r0 + kRows * warp + q;
            const uint4 *src = reinterpret_cast<const uint4 *>(w + (r * nb + b0) * 34);
#pragma unroll
            for (int u = 0; u < kWords; ++u) {
                const int i = lane + 32 * u;
                v[q][u] = (r < n && i < n16) ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
            }
        }
#pragma unroll
        for (int q = 0; q < kRows; ++q)
#pragma unroll
            for (int u = 0; u < kWords; ++u) {
                const int i = lane + 32 * u;
                if (i < n16) buf[kRows * warp + q][i] = v[q][u];
            }
        __syncwarp();
#pragma unroll
        for (int p = 0; p < kPairs; ++p) {
            const int pi = lane + 32 * p, rr = kRows * warp + pi / B, j = pi % B;
            const int64_t r = r0 + rr;
            float dw = 0.0f;
            if (r < n && j < cb) {
                // block j at byte 34j: its d at 34j, codes from 34j + 2; nine
                // words from the word holding byte 34j cover both
                const int base = (34 * j) >> 2, odd = j & 1;  // 34j % 4 == 2 for odd j
                const uint32_t *wd = reinterpret_cast<const uint32_t *>(buf[rr]) + base;
                uint32_t W[9];
#pragma unroll
                for (int u = 0; u < 9; ++u) W[u] = wd[u];
                dw = __half2float(
                    __ushort_as_half(static_cast<unsigned short>(odd ? (W[0] >> 16) : (W[0] & 0xffffu))));
                uint4 *dst = a16 + (r * nb + b0 + j) * 4;  // 64 bytes of f16 per block
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t q0 = odd ? W[2 * u + 1] : __byte_perm(W[2 * u], W[2 * u + 1], 0x5432);
                    const uint32_t q1 = odd ? W[2 * u + 2] : __byte_perm(W[2 * u + 1], W[2 * u + 2], 0x5432);
                    uint4 o;
                    q8::i8x4_to_f16x4(q0, o.x, o.y);
                    q8::i8x4_to_f16x4(q1, o.z, o.w);
                    dst[u] = o;
                }
            }
            sdw[j][dw_slot(rr)] = dw;  // rr < 32: its slot within the group
        }
        __syncthreads();
        const int64_t tile = r0 / BM;
        const int gbase = static_cast<int>(r0 - tile * BM);  // 0, 32, 64, 96: the group's first slot
        for (int i = threadIdx.x; i < cb * 32; i += NT)
            dwt[(tile * nb + b0 + (i >> 5)) * BM + gbase + (i & 31)] = sdw[i >> 5][i & 31];
        __syncthreads();  // sdw and buf are rewritten by the next item
    }
}

// Pre-pass over the activation: plane codes rows [0, t) -> f16 [t][k]
// (exact), and each block's d_a as f32 into dat[token tile][block][slot]
// in da_slot order (0 for tokens past t).
__global__ void __launch_bounds__(256)
gemm_prep_a_kernel(const uint4 *__restrict__ qs, const uint32_t *__restrict__ ds, int64_t t, int64_t k,
                   uint4 *__restrict__ b16, float *__restrict__ dat)
{
    q8::griddep_launch_dependents();
    q8::griddep_wait();  // the plane may come from the previous kernel
    const int64_t nb = k / 32;
    const int64_t chunks = t * (k / 16);  // 16-code chunks; qs row stride k: flat index
    const int64_t tiles = (t + BN - 1) / BN;
    const int64_t scales = tiles * nb * BN;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < chunks + scales;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        if (i < chunks) {
            const uint4 v = __ldg(qs + i);
            uint4 o0, o1;
            q8::i8x4_to_f16x4(v.x, o0.x, o0.y);
            q8::i8x4_to_f16x4(v.y, o0.z, o0.w);
            q8::i8x4_to_f16x4(v.z, o1.x, o1.y);
            q8::i8x4_to_f16x4(v.w, o1.z, o1.w);
            b16[2 * i] = o0;
            b16[2 * i + 1] = o1;
        } else {
            // slot s of (tile, block): the token column c with da_slot(c) == s
            const int64_t j = i - chunks;
            const int s = static_cast<int>(j % BN);
            const int64_t tb = j / BN;  // tile * nb + block
            const int64_t tile = tb / nb, b = tb - tile * nb;
            const int h = s >> 6, cg = (s >> 5) & 1, mm = (s >> 3) & 3, rp = (s >> 1) & 3, e = s & 1;
            const int c = 64 * h + 32 * cg + 8 * rp + 2 * mm + e;
            const int64_t tok = tile * BN + c;
            dat[j] = tok < t ? __half2float(__ushort_as_half(static_cast<unsigned short>(__ldg(ds + tok * nb + b) &
                                                                                          0xffffu)))
                             : 0.0f;
        }
    }
}

constexpr int kSplitSms = 152, kMaxSplits = 12, kMaxSplitsMany = 4;  // split-K bounds (see gemm_splits)

// Split-K: y = sum over z of part[z], added in z order (deterministic).
__global__ void __launch_bounds__(256)
gemm_split_reduce_kernel(const float *__restrict__ part, int splits, int64_t count, float *__restrict__ y)
{
    q8::griddep_launch_dependents();
    q8::griddep_wait();  // the partial tiles come from the GEMM just before
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i0 = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (count % 4 == 0) {  // four outputs per thread: 16-byte loads and stores (part and y are 16-byte aligned)
        const int64_t c4 = count / 4;
        const float4 *p4 = reinterpret_cast<const float4 *>(part);
        for (int64_t i = i0; i < c4; i += stride) {
            float4 pz[kMaxSplits];  // every split's loads in flight before the adds
#pragma unroll
            for (int z = 0; z < kMaxSplits; ++z)
                if (z < splits) pz[z] = __ldg(p4 + static_cast<int64_t>(z) * c4 + i);
            float4 v = pz[0];
#pragma unroll
            for (int z = 1; z < kMaxSplits; ++z)
                if (z < splits) v.x += pz[z].x, v.y += pz[z].y, v.z += pz[z].z, v.w += pz[z].w;
            reinterpret_cast<float4 *>(y)[i] = v;
        }
        return;
    }
    for (int64_t i = i0; i < count; i += stride) {
        float v = part[i];
        for (int z = 1; z < splits; ++z) v += part[static_cast<int64_t>(z) * count + i];
        y[i] = v;
    }
}

// How many CTAs share k (1 = none).  When the tiles alone leave most SMs idle
// (a few weight rows or tokens), k is split so that about one wave of CTAs
// runs, each over at least 4 stages (8 blocks).  With more tiles, k is split
// only when the last wave of whole tiles would leave enough SMs idle to pay
// for the partial tiles' traffic: a split s is scored by its waves of CTAs
// times a CTA's time (its stages plus a fixed ramp and store) plus the time to
// write and add the s partial tiles of every output, in the units of one
// stage of one CTA as measured on this kernel; the best score wins if it
// saves at least 3 % (e.g. 3584 x 18944 at t = 3325: 504 tiles fill 3.3
// waves, split 3 fills 9.9).  A fixed SM count is used so that the workspace
// size is a function of the shape alone; the first rule keeps splits * tiles
// at most that count, which bounds its partial tiles by about 15 MB, and the
// second allows at most 4 splits.
constexpr double kStageUs = 0.886;        // one stage (two blocks) of one CTA
constexpr double kCtaFixedUs = 4.0;       // a CTA's pipeline ramp and output store
constexpr double kPartialBytesPerUs = 6.5e6;  // partial tiles written and read back at about HBM rate
constexpr double kReduceLaunchUs = 3.0;
int gemm_splits(int64_t n, int64_t t, int64_t k)
{
    const int64_t tiles = ((n + BM - 1) / BM) * ((t + BN - 1) / BN);
    const int64_t nst = k / 32 / kStageBlocks;
    if (2 * tiles <= kSplitSms) {
        int64_t sp = kSplitSms / tiles;
        sp = sp > kMaxSplits ? kMaxSplits : sp;
        sp = sp > nst / 4 ? nst / 4 : sp;
        return sp < 1 ? 1 : static_cast<int>(sp);
    }
    auto score = [&](int64_t s) {
        const int64_t waves = (tiles * s + kSplitSms - 1) / kSplitSms;
        const int64_t stages = (nst + s - 1) / s;
        double us = static_cast<double>(waves) * (static_cast<double>(stages) * kStageUs + kCtaFixedUs);
        if (s > 1)  // the partials replace one f32 write of Y: 2s - 1 more passes over t x n f32
            us += static_cast<double>(2 * s - 1) * static_cast<double>(t) * static_cast<double>(n) * 4.0 /
                      kPartialBytesPerUs + kReduceLaunchUs;
        return us;
    };
    const double base = score(1);
    int best = 1;
    double best_us = base;
    for (int s = 2; s <= kMaxSplitsMany && nst / s >= 4; ++s) {
        const double us = score(s);
        if (us < best_us) {
            best_us = us;
            best = s;
        }
    }
    return best_us <= 0.97 * base ? best : 1;
}

// Workspace layout for (n, t, k): [f16 weights | f16 activation | d_w tiles |
// d_a tiles | partial tiles (split-K only: splits x t x n f32)].  With
// prepared weights (q8_0_gemm_prepared) the two weight parts live in the
// caller's prepared buffer instead, [f16 weights | d_w tiles], and the
// workspace holds the rest in the same order.
struct WsLayout {
    size_t a16, b16, dwt, dat, part, total;
    int splits;
};

size_t up1k(size_t v) { return (v + 1023) & ~static_cast<size_t>(1023); }

size_t dwt_bytes(int64_t n, int64_t k) { return static_cast<size_t>((n + BM - 1) / BM) * (k / 32) * BM * 4; }

WsLayout ws_layout(int64_t n, int64_t t, int64_t k, bool prepared = false)
{
    const size_t nb = static_cast<size_t>(k / 32);
    WsLayout L;
    L.splits = gemm_splits(n, t, k);
    L.a16 = 0;
    L.b16 = prepared ? 0 : up1k(L.a16 + static_cast<size_t>(n) * k * 2);
    L.dwt = up1k(L.b16 + static_cast<size_t>(t) * k * 2);
    L.dat = prepared ? L.dwt : up1k(L.dwt + dwt_bytes(n, k));
    L.part = up1k(L.dat + static_cast<size_t>((t + BN - 1) / BN) * nb * BN * 4);
    L.total = up1k(L.part + (L.splits > 1 ? static_cast<size_t>(L.splits) * t * n * 4 : 0));
    return L;
}

// Prepared weights: [f16 codes n x k | d_w tiles], the weight pre-pass's output.
size_t prep_w_dwt_offset(int64_t n, int64_t k) { return up1k(static_cast<size_t>(n) * k * 2); }
size_t prep_w_bytes(int64_t n, int64_t k) { return up1k(prep_w_dwt_offset(n, k) + dwt_bytes(n, k)); }

// The weight pre-pass: Q8_0 rows -> f16 codes [n][k] and d_w in tile order.
int launch_prep_w(const void *w, int64_t n, int64_t k, uint8_t *a16, float *dwt, cudaStream_t s)
{
    const int64_t nb = k / 32;
    const int sms = q8::device_sm_count();
    const int64_t pcap = static_cast<int64_t>(sms > 0 ? sms : 152) * 8;
    const int64_t groups = (n + BM - 1) / BM * (BM / 32);
    const int64_t wide = groups * ((nb + 31) / 32);  // items of 32 blocks
    const bool many = wide >= static_cast<int64_t>(sms > 0 ? sms : 152) * 4;
    const int64_t witems = many ? wide : groups * ((nb + 7) / 8);
    const unsigned wgrid = static_cast<unsigned>(witems < pcap ? witems : pcap);
    return many ? q8::launch_pdl(gemm_prep_w_kernel<32, 256>, dim3(wgrid), dim3(256), 0, s,
                                 static_cast<const uint8_t *>(w), n, static_cast<int>(nb),
                                 reinterpret_cast<uint4 *>(a16), dwt)
                : q8::launch_pdl(gemm_prep_w_kernel<8, 256>, dim3(wgrid), dim3(256), 0, s,
                                 static_cast<const uint8_t *>(w), n, static_cast<int>(nb),
                                 reinterpret_cast<uint4 *>(a16), dwt);
}

// The activation pre-pass, the GEMM and (split-K) the reduction, on weight
// operands already in the pre-pass's form.
int gemm_tc_core(const uint8_t *a16, const float *dwt, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds,
                 int64_t t, float *y, uint8_t *b16, float *dat, float *part, int splits, cudaStream_t s)
{
    const int64_t nb = k / 32;
    CUtensorMap ma, mb;
    if (!q8::make_map_2d(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT16, a16, static_cast<uint64_t>(k), static_cast<uint64_t>(n),
                         static_cast<uint64_t>(k * 2), 64, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !q8::make_map_2d(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT16, b16, static_cast<uint64_t>(k), static_cast<uint64_t>(t),
                         static_cast<uint64_t>(k * 2), 64, BN, CU_TENSOR_MAP_SWIZZLE_128B))
        return Q8_ERR_LAUNCH;
    const int sms = q8::device_sm_count();
    const int64_t pcap = static_cast<int64_t>(sms > 0 ? sms : 152) * 8;
    const int64_t awork = t * (k / 16) + (t + BN - 1) / BN * nb * BN;
    int64_t agrid = (awork + 255) / 256;
    agrid = agrid < pcap ? agrid : pcap;
    int st = q8::launch_pdl(gemm_prep_a_kernel, dim3(static_cast<unsigned>(agrid)), dim3(256), 0, s,
                            reinterpret_cast<const uint4 *>(qs), ds, t, k, reinterpret_cast<uint4 *>(b16), dat);
    if (st != Q8_OK) return st;
    const dim3 grid(static_cast<unsigned>((t + BN - 1) / BN), static_cast<unsigned>((n + BM - 1) / BM),
                    static_cast<unsigned>(splits));
    if (splits == 1) {
        if (!q8::set_max_dynamic_smem(reinterpret_cast<const void *>(gemm_tc_kernel<false>), kSmemBytes, 2))
            return Q8_ERR_LAUNCH;
        return q8::launch_pdl(gemm_tc_kernel<false>, grid, dim3(kThreads), kSmemBytes, s, ma, mb, dwt, dat, n, t,
                              static_cast<int>(nb), y, part);
    }
    if (!q8::set_max_dynamic_smem(reinterpret_cast<const void *>(gemm_tc_kernel<true>), kSmemBytes, 9))
        return Q8_ERR_LAUNCH;
    st = q8::launch_pdl(gemm_tc_kernel<true>, grid, dim3(kThreads), kSmemBytes, s, ma, mb, dwt, dat, n, t,
                        static_cast<int>(nb), y, part);
    if (st != Q8_OK) return st;
    const int64_t count = t * n;
    int64_t rgrid = (count % 4 == 0 ? count / 4 + 255 : count + 255) / 256;
    rgrid = rgrid < pcap ? rgrid : pcap;
    return q8::launch_pdl(gemm_split_reduce_kernel, dim3(static_cast<unsigned>(rgrid)), dim3(256), 0, s,
                          static_cast<const float *>(part), splits, count, y);
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

size_t gemm_workspace_bytes(int64_t n, int64_t t, int64_t k) { return ws_layout(n, t, k).total; }

size_t gemm_prepared_workspace_bytes(int64_t n, int64_t t, int64_t k) { return ws_layout(n, t, k, true).total; }

size_t gemm_prepared_weights_bytes(int64_t n, int64_t k) { return prep_w_bytes(n, k); }

// Requires k/32 % 8 == 0, 16-byte aligned pointers and a workspace of at least
// gemm_workspace_bytes(n, t, k) bytes (checked by the caller).
int gemm_tc_launch(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, int64_t t, float *y,
                   void *workspace, cudaStream_t s)
{
    const WsLayout L = ws_layout(n, t, k);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint8_t *a16 = ws + L.a16;
    float *dwt = reinterpret_cast<float *>(ws + L.dwt);
    const int st = launch_prep_w(w, n, k, a16, dwt, s);
    if (st != Q8_OK) return st;
    return gemm_tc_core(a16, dwt, n, k, qs, ds, t, y, ws + L.b16, reinterpret_cast<float *>(ws + L.dat),
                        reinterpret_cast<float *>(ws + L.part), L.splits, s);
}

// The weight pre-pass alone, into a caller's buffer of prep_w_bytes(n, k).
int gemm_prepare_weights_launch(const void *w, int64_t n, int64_t k, void *wprep, cudaStream_t s)
{
    uint8_t *p = static_cast<uint8_t *>(wprep);
    return launch_prep_w(w, n, k, p, reinterpret_cast<float *>(p + prep_w_dwt_offset(n, k)), s);
}

// The GEMM on prepared weights: the activation pre-pass, the GEMM and (split-K)
// the reduction; the workspace is gemm_prepared_workspace_bytes(n, t, k).
int gemm_tc_prepared_launch(const void *wprep, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, int64_t t,
                            float *y, void *workspace, cudaStream_t s)
{
    const WsLayout L = ws_layout(n, t, k, true);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const uint8_t *p = static_cast<const uint8_t *>(wprep);
    return gemm_tc_core(p, reinterpret_cast<const float *>(p + prep_w_dwt_offset(n, k)), n, k, qs, ds, t, y,
                        ws + L.b16, reinterpret_cast<float *>(ws + L.dat), reinterpret_cast<float *>(ws + L.part),
                        L.splits, s);
}

} // namespace q8

// ---------------------------------------------------------------------------
// q8_0_gemm_noalloc: the same GEMM with its scratch in a fixed device array.
//
// Some callers cannot allocate device memory on the way to this call: a
// serving engine that reserved all of the GPU's memory for its own pool at
// start-up, a plugin whose host forbids allocation once it is initialised,
// or a latency-critical path that cannot afford cudaMalloc's implicit
// synchronisation.  For them the prepared operands live in the array
// below.  It is part of the library's device image, so every GPU on which
// this library's GEMM module is loaded keeps these bytes until the process
// exits, whether or not this entry point is ever called.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(32) << 20;  // 32 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64];      // device address of g_noalloc_scratch, per device ordinal
CUcontext g_noalloc_ctx[64];  // the context that address belongs to

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

// cuCtxGetCurrent through the runtime's driver entry point (the library does
// not link libcuda); looked up once.
CtxGetCurrentFn ctx_get_current_fn()
{
    static const CtxGetCurrentFn fn = []() -> CtxGetCurrentFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<CtxGetCurrentFn>(p);
        return nullptr;
    }();
    return fn;
}

// Device address of the scratch array on the current device (the array's
// name in host code is only a stand-in for it).  It is looked up on the first
// call on a device and again whenever the current context is not the one it
// was looked up in (after a device reset the module is loaded anew and the
// array may sit elsewhere).
int noalloc_scratch(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return Q8_ERR_DEVICE;
    CtxGetCurrentFn get_ctx = ctx_get_current_fn();
    CUcontext ctx = nullptr;
    if (!get_ctx || get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return Q8_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev] || g_noalloc_ctx[dev] != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return Q8_ERR_CUDA;
        g_noalloc_ptr[dev] = p;
        g_noalloc_ctx[dev] = ctx;
    }
    *out = g_noalloc_ptr[dev];
    return Q8_OK;
}

} // namespace

extern "C" int q8_0_gemm_noalloc(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds,
                                 int64_t t, int64_t rows_pad, float *y, void *stream)
{
    if (!w || !qs || !ds || !y || n < 1 || t < 1 || k <= 0 || (k % 32) != 0 || rows_pad < t) return Q8_ERR_ARG;
    const size_t need = q8_0_gemm_workspace_bytes(n, t, k);
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
    if (t <= q8::kSlicedMaxTokens) return q8::gemv_sliced_launch(w, n, k, qs, ds, y, t, s);
    if (n > int64_t(65535) * 128 || t > (int64_t(1) << 31) - 256 || k > (int64_t(1) << 31) / 2) return Q8_ERR_ARG;
    void *scratch = nullptr;
    const int st = noalloc_scratch(&scratch);
    if (st != Q8_OK) return st;
    return q8::gemm_tc_launch(w, n, k, qs, ds, t, y, scratch, s);
}

extern "C" size_t q8_0_gemm_noalloc_max_bytes(void) { return kNoAllocScratchBytes; }

