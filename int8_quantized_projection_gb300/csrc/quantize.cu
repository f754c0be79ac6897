// quantize.cu -- q8_0 activation quantization, standalone and fused into its
// producers (RMSNorm, SwiGLU).
//
// All three kernels are HBM-bound streams.  They share one register-level
// encoder (q8::q8_encode8): a warp reads 32 consecutive float4, so 8 adjacent
// lanes hold one 32-element block and amax / ssum are 3-step shuffle
// reductions.  The fused kernels encode the f32 values they have just
// computed, straight from registers: the page's producer-fused kernels
// ("54 - r51 - producer-fused A-quantize mode 1", sec. 3.1) re-read their
// f32 output from L1/L2 because their phase-1 lane mapping did not line up
// with one-thread-per-block quantization; here both phases use the same
// lane mapping, so no re-read is needed and the plane is still the exact
// encoding of the stored f32 output.
#include "q8_common.cuh"

namespace {

__device__ unsigned int g_quant_err;

constexpr int kQuantThreads = 256;
constexpr int kQuantUnroll = 4;  // float4 loads in flight per lane

// Streaming 16-byte load that does not allocate in L1.
__device__ __forceinline__ float4 ld_stream(const float4 *p)
{
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// --------------------------------------------------------------------------
// quantize_q8_0: flat stream over the [rows][k] f32 array.  Because k % 32 ==
// 0, the flat float4 index f maps to qs word f and to ds word f/8; rows past
// `rows` (up to rows_pad) are the zero tail.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(kQuantThreads)
quantize_q8_0_kernel(const float4 *__restrict__ x, int64_t n4_valid, int64_t n4_total,
                     uint32_t *__restrict__ qs, uint32_t *__restrict__ ds)
{
    q8::griddep_launch_dependents();  // consumers may start their prologue
    q8::griddep_wait();               // inputs may come from the previous kernel
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    // Each warp iteration covers kQuantUnroll chunks of 32 float4 (4 blocks each).
    for (int64_t base = warp * 32 * kQuantUnroll; base < n4_total; base += nwarps * 32 * kQuantUnroll) {
        float4 v[kQuantUnroll];
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int64_t f = base + u * 32 + lane;
            v[u] = (f < n4_valid) ? ld_stream(x + f) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int64_t f = base + u * 32 + lane;
            const q8::Q8Enc e = q8::q8_encode8(v[u]);  // tail rows encode zeros -> all-zero words
            if (f < n4_total) {
                qs[f] = e.qword;
                if ((lane & 7) == 0) ds[f >> 3] = e.dsword;
            }
        }
    }
}

// --------------------------------------------------------------------------
// rmsnorm_quant: persistent CTAs, one token row at a time; each thread keeps
// J float4 of the row in registers (float4 index f = tid + j*blockDim) and
// prefetches its share of the CTA's next row before reducing the current one,
// so x is read once, y written once and the plane encoded from the same
// registers.  "54 - r51 - producer-fused A-quantize mode 1", sec. 3.2:
// ss = sum x^2, scale = rsqrt(ss/d + eps), y = (x * scale) * w.
// --------------------------------------------------------------------------
// widest row whose weight vector is staged in shared memory (32 KB: below the
// 48 KB a kernel may use without opting in)
constexpr int kNormSmemMax = 8192;

template <int J>
__global__ void __launch_bounds__(512)
rmsnorm_quant_kernel(const float *__restrict__ x, const float *__restrict__ w, float eps,
                     float *__restrict__ y, int64_t rows, int64_t rows_pad, int d,
                     uint32_t *__restrict__ qs, uint32_t *__restrict__ ds)
{
    __shared__ float red[2][32];
    extern __shared__ float4 wsm[];   // the weight vector, when it is staged (d <= kNormSmemMax)
    const int F = d >> 2;
    const int P = blockDim.x;
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int nw = P >> 5;
    const bool staged = d <= kNormSmemMax;
    const float4 *w4 = reinterpret_cast<const float4 *>(w);
    q8::griddep_launch_dependents();  // consumers may start their prologue
    // The weight vector is a constant input, the same for every row: stage it
    // in shared memory before waiting for the previous kernel, so a row costs
    // one memory round trip (its own) instead of two.  Ordered before its
    // first use by the barrier in the first row's reduction.
    if (staged)
        for (int f = tid; f < F; f += P) wsm[f] = __ldg(w4 + f);
    q8::griddep_wait();               // inputs may come from the previous kernel

    auto load_row = [&](int64_t t, float4 (&v)[J]) {
        const float4 *xr = reinterpret_cast<const float4 *>(x + t * static_cast<int64_t>(d));
#pragma unroll
        for (int j = 0; j < J; ++j) {
            const int f = tid + j * P;
            v[j] = (t < rows && f < F) ? ld_stream(xr + f) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };

    float4 v[J], vn[J];
    int64_t t = blockIdx.x;
    load_row(t, v);
    for (int it = 0; t < rows_pad; ++it, t += gridDim.x) {
        const int64_t tn = t + gridDim.x;
        load_row(tn, vn);  // next row in flight while this one is reduced and written
        uint32_t *qrow = qs + t * F;
        uint32_t *drow = ds + t * (F >> 3);
        if (t >= rows) {  // padded token row: zero plane row
            for (int f = tid; f < F; f += P) {
                qrow[f] = 0u;
                if ((f & 7) == 0) drow[f >> 3] = 0u;
            }
        } else {
            float ss = 0.0f;
#pragma unroll
            for (int j = 0; j < J; ++j) ss = q8::rms_sumsq4(ss, v[j]);
            ss = q8::rms_warp_sum(ss);
            float *rb = red[it & 1];  // alternate buffers: one barrier per row suffices
            if (lane == 0) rb[tid >> 5] = ss;
            __syncthreads();
            float tot = 0.0f;
            for (int i = 0; i < nw; ++i) tot += rb[i];  // same fixed order in every thread
            const float scale = q8::rms_scale(tot, d, eps);
            float4 *yr = reinterpret_cast<float4 *>(y + t * static_cast<int64_t>(d));
#pragma unroll
            for (int j = 0; j < J; ++j) {
                const int f = tid + j * P;
                const bool ok = f < F;  // uniform over each 8-lane block group
                float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
                if (ok) {
                    o = q8::rms_apply4(v[j], scale, staged ? wsm[f] : __ldg(w4 + f));
                    if (y) yr[f] = o;  // mode 2 (y == NULL): the f32 output is dead, only the plane is written
                }
                const q8::Q8Enc e = q8::q8_encode8(o);
                if (ok) {
                    qrow[f] = e.qword;
                    if ((lane & 7) == 0) drow[f >> 3] = e.dsword;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < J; ++j) v[j] = vn[j];
    }
}

// --------------------------------------------------------------------------
// rmsnorm_quant for many rows (more than one per SM) of moderate width: one
// persistent CTA per SM made of row groups of four warps.  A group owns a row
// at a time; its rows arrive by TMA into the group's two shared-memory slots,
// the next while it works on the current one, so each SM keeps a dozen rows
// in flight and no group waits for another (a group meets once per row on a
// named barrier of its own, to add its warps' sums of squares; each warp then
// releases the row's slot through an mbarrier that the thread refilling the
// slot waits on, so the other warps go on to the next row).  Thread b of a
// group owns the row's 32-element block b whole: its amax and code sum are
// register reductions and its d and 1/d are computed once, so the encoder
// costs a fraction of the per-lane (8 lanes per block) form.  Per row: each
// thread sums the squares of its block (two partial sums, even and odd
// elements), the warps reduce by xor shuffles and their four sums are added
// in warp order; then scale, write y (mode 1) and encode.  The kernel is
// bound by instruction issue rather than by DRAM, so the arithmetic runs two
// elements per instruction where it can (packed f32x2 sums of squares,
// scaling and code products, three-input maxima) and the codes are rounded
// by an add on the FMA pipe instead of one conversion per element; every
// element still takes the same roundings as the scalar form.
//
// A row is loaded as a 3-D tensor box [1 row][d/32 blocks][32 floats] with
// the 128-byte swizzle: block b's 16-byte chunk c lands at chunk c ^ (b mod 8)
// of its 128-byte line (slots start on 1024-byte boundaries, so the line's
// address bits 7..9 are b mod 8).  Thread b reads its chunk c from there into
// register c, so the eight threads of a quarter warp hit eight different bank
// groups while every register index stays static, and the block's 32 codes
// leave as two 16-byte stores.  The weight vector is staged once per CTA in
// the same swizzled order.
// --------------------------------------------------------------------------
constexpr int kGrpThreads = 128;     // four warps per row, one block per thread
constexpr int kGrpSlots = 2;         // row slots per group
constexpr int kGrpMax = 8;           // groups per CTA (1024 threads)
constexpr int kGrpMaxNorm = 6;       // RMSNorm groups per CTA (768 threads: up to 80 registers a thread)
constexpr int kGrpSmemBudget = 200 * 1024;  // weight vector + every group's slots
constexpr int kGrpMaxD = 32 * kGrpThreads;  // 4096: one block per thread

// bytes of one row slot (and of the staged weight vector): d floats, rounded
// up to whole 1024-byte swizzle atoms
int rowgroup_slot_bytes(int d) { return (d * 4 + 1023) / 1024 * 1024; }

int rowgroup_groups(int d, bool norm)
{
    const int per = rowgroup_slot_bytes(d);
    const int g = (kGrpSmemBudget - (norm ? per : 0)) / (per * kGrpSlots);
    return g > kGrpMax ? kGrpMax : g;
}

// dynamic shared memory of a launch: 1024 bytes of alignment slack, the
// weight vector (RMSNorm) and every group's slots
size_t rowgroup_smem(int d, bool norm, int groups)
{
    const size_t per = static_cast<size_t>(rowgroup_slot_bytes(d));
    return 1024 + (norm ? per : 0) + per * kGrpSlots * groups;
}

__device__ __forceinline__ void group_sync(int id)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(kGrpThreads) : "memory");
}

// Maximum of three floats in one instruction (the three-input max.f32 of
// the sm_100 family).
__device__ __forceinline__ float max3f(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// The body shared by RMSNorm + quantize (kNorm) and the plain quantizer
// (rows of x encoded as they are: no sum of squares, weight or y).
// tmx: x as [rows][d/32][32] f32, box {32, d/32, 1}, 128-byte swizzle.
template <bool kNorm>
__device__ __forceinline__ void rowgroup_body(const CUtensorMap *tmx, const float *__restrict__ w, float eps,
                                              float *__restrict__ y, int64_t rows, int64_t rows_pad, int d,
                                              uint32_t *__restrict__ qs, uint32_t *__restrict__ ds)
{
    extern __shared__ __align__(128) uint8_t smem_rg[];
    __shared__ __align__(8) uint64_t full[kGrpMax * kGrpSlots];
    __shared__ __align__(8) uint64_t empty[kGrpMax * kGrpSlots];  // the group's four warps are done with a slot
    __shared__ float red[kGrpMax][2][kGrpThreads / 32];
    __shared__ int okf[kGrpMax][2][kGrpThreads / 32];
    const int F = d >> 2, nb = d >> 5;
    const int grp = threadIdx.x / kGrpThreads, gt = threadIdx.x % kGrpThreads;
    const int lane = gt & 31, gw = gt >> 5;
    const int ngroups = blockDim.x / kGrpThreads;
    const uint32_t raw = q8::smem_u32(smem_rg);
    uint8_t *base = smem_rg + (((raw + 1023u) & ~1023u) - raw);  // 1024-byte aligned
    const int slot_f4 = ((d * 4 + 1023) / 1024 * 1024) / 16;      // float4 per slot
    const float4 *wsm = reinterpret_cast<const float4 *>(base);
    float4 *myslots = reinterpret_cast<float4 *>(base) + static_cast<int64_t>(slot_f4) * ((kNorm ? 1 : 0) + kGrpSlots * grp);
    uint64_t *mybar = full + kGrpSlots * grp;
    uint64_t *myempty = empty + kGrpSlots * grp;
    const uint32_t row_bytes = static_cast<uint32_t>(d) * 4u;  // the box's bytes
    const bool mine_blk = gt < nb;                             // this thread's block exists
    const int sw = gt & 7;                                     // chunk c of block gt sits at c ^ sw
    q8::griddep_launch_dependents();  // consumers may start their prologue
    // the weight vector is a constant input: staged (swizzled like the rows)
    // before the dependency wait
    if (kNorm)
        for (int f = threadIdx.x; f < F; f += blockDim.x)
            reinterpret_cast<float4 *>(base)[(f & ~7) | ((f ^ (f >> 3)) & 7)] =
                __ldg(reinterpret_cast<const float4 *>(w) + f);
    if (gt == 0) {
        for (int s = 0; s < kGrpSlots; ++s) {
            q8::mbar_init(&mybar[s], 1);
            q8::mbar_init(&myempty[s], kGrpThreads / 32);
        }
        q8::fence_mbar_init();
    }
    __syncthreads();
    q8::griddep_wait();  // x may come from the previous kernel

    // this group's rows: t = g0 + i * stride, dealt round-robin over the CTAs
    // first (row t to CTA t mod the grid), so every SM gets the same number
    // of rows to within one; rows at or past `rows` (the zero tail, all at
    // the end) are not loaded
    const int64_t g0 = static_cast<int64_t>(blockIdx.x) + static_cast<int64_t>(grp) * gridDim.x;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * ngroups;
    const int64_t mine = g0 < rows_pad ? (rows_pad - g0 + stride - 1) / stride : 0;
    int64_t issued = 0;  // thread gt == 0: rows whose load has been issued (or that need none)
    auto issue_upto = [&](int64_t upto) {
        for (; issued < upto && issued < mine; ++issued) {
            const int64_t t = g0 + issued * stride;
            if (t >= rows) continue;
            const int s = static_cast<int>(issued % kGrpSlots);
            if (issued >= kGrpSlots) {
                // the row that used this slot before must be read by all four warps
                if (!q8::mbar_wait_bounded(&myempty[s], static_cast<uint32_t>((issued - kGrpSlots) / kGrpSlots) & 1u)) {
                    atomicOr(&g_quant_err, 1u);
                    break;
                }
                q8::fence_proxy_async_smem();  // those reads come before the copy into the slot
            }
            q8::mbar_arrive_expect_tx(&mybar[s], row_bytes);
            q8::tma_load_3d(q8::smem_u32(myslots + static_cast<int64_t>(s) * slot_f4), tmx, 0, 0,
                            static_cast<int>(t), q8::smem_u32(&mybar[s]));
        }
    };
    if (gt == 0) issue_upto(kGrpSlots);
    int64_t i = 0;
    for (; i < mine; ++i) {
        const int64_t t = g0 + i * stride;
        uint4 *qrow = reinterpret_cast<uint4 *>(qs + t * F);  // 32 codes = two uint4 per block
        uint32_t *drow = ds + t * nb;
        if (t >= rows) {  // padded token row: zero plane row
            if (mine_blk) {
                qrow[2 * gt] = make_uint4(0u, 0u, 0u, 0u);
                qrow[2 * gt + 1] = make_uint4(0u, 0u, 0u, 0u);
                drow[gt] = 0u;
            }
            continue;
        }
        const int s = static_cast<int>(i % kGrpSlots);
        const bool got = q8::mbar_wait_bounded(&mybar[s], static_cast<uint32_t>(i / kGrpSlots) & 1u);
        const float4 *xb = myslots + static_cast<int64_t>(s) * slot_f4 + 8 * gt;
        float4 v[8];
        float ss = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = (got && mine_blk) ? xb[k ^ sw] : make_float4(0.f, 0.f, 0.f, 0.f);
        if (kNorm) {
            // two partial sums (even and odd elements), one packed FMA per pair
            float2 s2 = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float2 lo = make_float2(v[k].x, v[k].y), hi = make_float2(v[k].z, v[k].w);
                s2 = __ffma2_rn(lo, lo, s2);
                s2 = __ffma2_rn(hi, hi, s2);
            }
            ss = q8::rms_warp_sum(s2.x + s2.y);
        }
        const int rb = static_cast<int>(i & 1);  // alternate buffers: one exchange barrier per row suffices
        const bool all_got = __all_sync(Q8_FULL_MASK, got);
        if (lane == 0) {
            red[grp][rb][gw] = ss;
            okf[grp][rb][gw] = all_got ? 1 : 0;
        }
        group_sync(1 + grp);
        bool all_ok = true;
        float tot = 0.0f;
#pragma unroll
        for (int k = 0; k < kGrpThreads / 32; ++k) {
            tot += red[grp][rb][k];  // same fixed order in every thread
            all_ok = all_ok && okf[grp][rb][k] != 0;
        }
        if (!all_ok) {  // a load did not arrive in time: report, stop (the whole group alike)
            if (gt == 0) atomicOr(&g_quant_err, 1u);
            break;
        }
        if (mine_blk) {
            float amax = 0.0f;
            if (kNorm) {
                const float scale = q8::rms_scale(tot, d, eps);
                const float4 *wb = wsm + 8 * gt;
                const float2 sc2 = make_float2(scale, scale);
#pragma unroll
                for (int k = 0; k < 8; ++k) {  // (x * scale) * w, two roundings per element, two elements per op
                    const float4 wv = wb[k ^ sw];
                    const float2 lo = __fmul2_rn(__fmul2_rn(make_float2(v[k].x, v[k].y), sc2), make_float2(wv.x, wv.y));
                    const float2 hi = __fmul2_rn(__fmul2_rn(make_float2(v[k].z, v[k].w), sc2), make_float2(wv.z, wv.w));
                    v[k] = make_float4(lo.x, lo.y, hi.x, hi.y);
                }
                if (y) {  // mode 2 (y == NULL): only the plane is written
                    float4 *yb = reinterpret_cast<float4 *>(y + t * static_cast<int64_t>(d)) + 8 * gt;
#pragma unroll
                    for (int k = 0; k < 8; ++k) yb[k] = v[k];
                }
            }
            {
                float m[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    m[k] = max3f(fabsf(v[k].x), fabsf(v[k].y), fabsf(v[k].z));
                    m[k] = fmaxf(m[k], fabsf(v[k].w));
                }
                amax = max3f(max3f(m[0], m[1], m[2]), max3f(m[3], m[4], m[5]), fmaxf(m[6], m[7]));
            }
            const float dq = q8::q8_block_d(amax);
            const float di = q8::q8_block_di(dq);
            uint32_t qw[8];
            int sum = 0;
            if (q8::block_rounds_by_add(dq)) {
                uint32_t bsum = 0u;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    uint32_t b0, b1, b2, b3;
                    q8::round_by_add2(v[k].x, v[k].y, di, b0, b1);
                    q8::round_by_add2(v[k].z, v[k].w, di, b2, b3);
                    bsum += b0 + b1 + b2 + b3;
                    qw[k] = q8::pack4(static_cast<int>(b0), static_cast<int>(b1), static_cast<int>(b2),
                                      static_cast<int>(b3));
                }
                sum = static_cast<int>(bsum - 32u * q8::kRoundMagicBits);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int c0 = q8::q8_code(v[k].x, di), c1 = q8::q8_code(v[k].y, di);
                    const int c2 = q8::q8_code(v[k].z, di), c3 = q8::q8_code(v[k].w, di);
                    sum += c0 + c1 + c2 + c3;
                    qw[k] = q8::pack4(c0, c1, c2, c3);
                }
            }
            qrow[2 * gt] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
            qrow[2 * gt + 1] = make_uint4(qw[4], qw[5], qw[6], qw[7]);
            drow[gt] = q8::q8_dsword(dq, sum);
        }
        __syncwarp();
        if (lane == 0) q8::mbar_arrive(&myempty[s]);  // this warp is done with the row's slot
        if (gt == 0) issue_upto(i + 1 + kGrpSlots);
    }
    // after a timeout, let this group's loads still in flight land before it exits
    if (gt == 0)
        for (int64_t k = i; k < issued; ++k)
            if (g0 + k * stride < rows)
                (void)q8::mbar_wait_bounded(&mybar[k % kGrpSlots], static_cast<uint32_t>(k / kGrpSlots) & 1u,
                                            Q8_DRAIN_LIMIT_NS);
}

__global__ void __launch_bounds__(kGrpThreads * kGrpMaxNorm, 1)
rmsnorm_quant_rowgroup_kernel(const __grid_constant__ CUtensorMap tmx, const float *__restrict__ w, float eps,
                              float *__restrict__ y, int64_t rows, int64_t rows_pad, int d,
                              uint32_t *__restrict__ qs, uint32_t *__restrict__ ds)
{
    rowgroup_body<true>(&tmx, w, eps, y, rows, rows_pad, d, qs, ds);
}

__global__ void __launch_bounds__(kGrpThreads * kGrpMax, 1)
quantize_q8_0_rowgroup_kernel(const __grid_constant__ CUtensorMap tmx, int64_t rows, int64_t rows_pad, int d,
                              uint32_t *__restrict__ qs, uint32_t *__restrict__ ds)
{
    rowgroup_body<false>(&tmx, nullptr, 0.0f, nullptr, rows, rows_pad, d, qs, ds);
}

// x as the row-group kernels' TMA source: [rows][d/32][32] f32, one row per box
bool rowgroup_x_map(CUtensorMap *m, const float *x, int64_t rows, int d)
{
    return q8::make_map_3d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, x, 32, static_cast<uint64_t>(d / 32),
                           static_cast<uint64_t>(rows), 128, static_cast<uint64_t>(d) * 4, 32,
                           static_cast<uint32_t>(d / 32), 1, CU_TENSOR_MAP_SWIZZLE_128B);
}

// --------------------------------------------------------------------------
// swiglu_quant: flat elementwise stream, y = g / (1 + exp(-g)) * u
// ("54 - r51 - producer-fused A-quantize mode 1", sec. 3.2), encoded from
// registers into the plane in the same pass.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(kQuantThreads)
swiglu_quant_kernel(const float4 *__restrict__ g, const float4 *__restrict__ u, float4 *__restrict__ y,
                    int64_t n4_valid, int64_t n4_total, uint32_t *__restrict__ qs, uint32_t *__restrict__ ds)
{
    q8::griddep_launch_dependents();  // consumers may start their prologue
    q8::griddep_wait();               // inputs may come from the previous kernel
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    constexpr int U = 4;  // float4 pairs in flight per lane (2: 104 us at 3325 x 18944, 4: 91 us, 8 spills)
    for (int64_t base = warp * 32 * U; base < n4_total; base += nwarps * 32 * U) {
        float4 gv[U], uv[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t f = base + k * 32 + lane;
            const bool ok = f < n4_valid;
            gv[k] = ok ? ld_stream(g + f) : make_float4(0.f, 0.f, 0.f, 0.f);
            uv[k] = ok ? ld_stream(u + f) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t f = base + k * 32 + lane;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
            if (f < n4_valid) {
                o = q8::silu_mul4(gv[k], uv[k]);
                if (y) y[f] = o;  // mode 2 (y == NULL): the f32 output is dead, only the plane is written
            }
            const q8::Q8Enc e = q8::q8_encode8(o);
            if (f < n4_total) {
                qs[f] = e.qword;
                if ((lane & 7) == 0) ds[f >> 3] = e.dsword;
            }
        }
    }
}

int flat_grid(int64_t n4_total, int per_warp_iter)
{
    const int64_t warps = (n4_total + 32 * per_warp_iter - 1) / (32 * per_warp_iter);
    const int64_t ctas = (warps + (kQuantThreads / 32) - 1) / (kQuantThreads / 32);
    const int sms = q8::device_sm_count();
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 152) * 8;  // 8 resident CTAs per SM
    return static_cast<int>(ctas < cap ? (ctas > 0 ? ctas : 1) : cap);
}

int check_plane_args(int64_t rows, int64_t k, const void *qs, const void *ds, int64_t rows_pad)
{
    if (!qs || !ds) return Q8_ERR_ARG;
    if (rows < 0 || k <= 0 || (k % 32) != 0 || rows_pad < rows || rows_pad < 1) return Q8_ERR_ARG;
    if (!q8::aligned16(qs) || !q8::aligned16(ds)) return Q8_ERR_ALIGN;
    return Q8_OK;
}

} // namespace

extern "C" int quantize_q8_0(const float *x, int64_t rows, int64_t k, int8_t *qs, uint32_t *ds,
                             int64_t rows_pad, void *stream)
{
    if (rows > 0 && !x) return Q8_ERR_ARG;
    int st = check_plane_args(rows, k, qs, ds, rows_pad);
    if (st != Q8_OK) return st;
    if (rows > 0 && !q8::aligned16(x)) return Q8_ERR_ALIGN;
    if (!q8::device_is_sm103()) return Q8_ERR_DEVICE;
    const int sms = q8::device_sm_count();
    const int nsm = sms > 0 ? sms : 152;
    // two CTAs per SM, each with half the groups that fit: an SM takes the next
    // launch's first CTA as soon as one of them ends (the norm kernel keeps one
    // CTA per SM: a second copy of its weight vector costs more than that gains)
    const int ng = k <= kGrpMaxD ? rowgroup_groups(static_cast<int>(k), false) / 2 : 0;
    if (rows_pad > nsm && ng >= 2 && rows < (int64_t(1) << 31)) {
        // many rows: row groups streaming the rows through shared memory
        const size_t smem = rowgroup_smem(static_cast<int>(k), false, ng);
        CUtensorMap mx{};
        if (rows > 0 && !rowgroup_x_map(&mx, x, rows, static_cast<int>(k))) return Q8_ERR_LAUNCH;
        if (!q8::set_max_dynamic_smem(reinterpret_cast<const void *>(quantize_q8_0_rowgroup_kernel),
                                      static_cast<int>(smem), 13))
            return Q8_ERR_LAUNCH;
        return q8::launch_pdl(quantize_q8_0_rowgroup_kernel, dim3(static_cast<unsigned>(2 * nsm)),
                              dim3(kGrpThreads * ng), smem, static_cast<cudaStream_t>(stream), mx, rows, rows_pad,
                              static_cast<int>(k), reinterpret_cast<uint32_t *>(qs), ds);
    }
    const int64_t n4_valid = rows * k / 4, n4_total = rows_pad * k / 4;
    return q8::launch_pdl(quantize_q8_0_kernel, dim3(flat_grid(n4_total, kQuantUnroll)), dim3(kQuantThreads), 0,
                          static_cast<cudaStream_t>(stream), reinterpret_cast<const float4 *>(x), n4_valid, n4_total,
                          reinterpret_cast<uint32_t *>(qs), ds);
}

extern "C" int rmsnorm_quant(const float *x, const float *w, float eps, float *y, int64_t rows, int64_t d,
                             int8_t *qs, uint32_t *ds, int64_t rows_pad, void *stream)
{
    if (rows > 0 && (!x || !w)) return Q8_ERR_ARG;  // y may be NULL (mode 2)
    int st = check_plane_args(rows, d, qs, ds, rows_pad);
    if (st != Q8_OK) return st;
    if (d > 32768) return Q8_ERR_ARG;  // row held in registers: at most 16 float4 x 512 threads
    if (rows > 0 && (!q8::aligned16(x) || !q8::aligned16(w) || (y && !q8::aligned16(y)))) return Q8_ERR_ALIGN;
    if (!q8::device_is_sm103()) return Q8_ERR_DEVICE;
    const int F = static_cast<int>(d / 4);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int sms = q8::device_sm_count();
    const int nsm = sms > 0 ? sms : 152;
    uint32_t *q32 = reinterpret_cast<uint32_t *>(qs);
    const int di = static_cast<int>(d);
    const int ng = rowgroup_groups(di, true) < kGrpMaxNorm ? rowgroup_groups(di, true) : kGrpMaxNorm;
    if (rows_pad > nsm && d <= kGrpMaxD && ng >= 2 && rows < (int64_t(1) << 31)) {
        // many rows: row groups streaming their rows through shared memory, one CTA per SM
        const size_t smem = rowgroup_smem(di, true, ng);
        CUtensorMap mx{};
        if (rows > 0 && !rowgroup_x_map(&mx, x, rows, di)) return Q8_ERR_LAUNCH;
        if (!q8::set_max_dynamic_smem(reinterpret_cast<const void *>(rmsnorm_quant_rowgroup_kernel),
                                      static_cast<int>(smem), 12))
            return Q8_ERR_LAUNCH;
        return q8::launch_pdl(rmsnorm_quant_rowgroup_kernel, dim3(static_cast<unsigned>(nsm)), dim3(kGrpThreads * ng),
                              smem, s, mx, w, eps, y, rows, rows_pad, di, q32, ds);
    }
    // float4 per thread: up to 256 threads per row when CTAs take several rows
    // (four CTAs per SM keep four rows in flight), up to 512 when every CTA
    // has at most one row (a decode token: shorter chains per thread)
    const int max_p = rows_pad <= (sms > 0 ? sms : 152) ? q8::kRmsMaxThreadsOneRow : q8::kRmsMaxThreadsManyRows;
    int J, P;
    q8::rms_row_mapping(F, max_p, J, P);
    // persistent grid: enough CTAs to fill the SMs (registers allow ~4 per SM
    // at these block sizes), each walking rows with a stride of the grid
    const int64_t per_sm = P <= 256 ? 4 : 2;
    const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 152) * per_sm;
    const dim3 grid(static_cast<unsigned>(rows_pad < cap ? rows_pad : cap));
    const size_t wsmem = d <= kNormSmemMax ? static_cast<size_t>(d) * 4 : 0;
    switch (J) {
    case 1: return q8::launch_pdl(rmsnorm_quant_kernel<1>, grid, dim3(P), wsmem, s, x, w, eps, y, rows, rows_pad, di, q32, ds);
    case 2: return q8::launch_pdl(rmsnorm_quant_kernel<2>, grid, dim3(P), wsmem, s, x, w, eps, y, rows, rows_pad, di, q32, ds);
    case 4: return q8::launch_pdl(rmsnorm_quant_kernel<4>, grid, dim3(P), wsmem, s, x, w, eps, y, rows, rows_pad, di, q32, ds);
    case 8: return q8::launch_pdl(rmsnorm_quant_kernel<8>, grid, dim3(P), wsmem, s, x, w, eps, y, rows, rows_pad, di, q32, ds);
    default: return q8::launch_pdl(rmsnorm_quant_kernel<16>, grid, dim3(P), wsmem, s, x, w, eps, y, rows, rows_pad, di, q32, ds);
    }
}

extern "C" int swiglu_quant(const float *gate, const float *up, float *y, int64_t rows, int64_t nf, int8_t *qs,
                            uint32_t *ds, int64_t rows_pad, void *stream)
{
    if (rows > 0 && (!gate || !up)) return Q8_ERR_ARG;  // y may be NULL (mode 2)
    int st = check_plane_args(rows, nf, qs, ds, rows_pad);
    if (st != Q8_OK) return st;
    if (rows > 0 && (!q8::aligned16(gate) || !q8::aligned16(up) || (y && !q8::aligned16(y)))) return Q8_ERR_ALIGN;
    if (!q8::device_is_sm103()) return Q8_ERR_DEVICE;
    const int64_t n4_valid = rows * nf / 4, n4_total = rows_pad * nf / 4;
    return q8::launch_pdl(swiglu_quant_kernel, dim3(flat_grid(n4_total, 4)), dim3(kQuantThreads), 0,
                          static_cast<cudaStream_t>(stream), reinterpret_cast<const float4 *>(gate),
                          reinterpret_cast<const float4 *>(up), reinterpret_cast<float4 *>(y), n4_valid, n4_total,
                          reinterpret_cast<uint32_t *>(qs), ds);
}

namespace q8 {

int quant_take_error(cudaStream_t s)
{
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_quant_err, sizeof(v), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_quant_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return Q8_ERR_CUDA;
    return v ? Q8_ERR_DEVICE_TIMEOUT : Q8_OK;
}

} // namespace q8
