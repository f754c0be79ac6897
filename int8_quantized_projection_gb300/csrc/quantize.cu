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
    constexpr int U = 2;
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
    uint32_t *q32 = reinterpret_cast<uint32_t *>(qs);
    const int di = static_cast<int>(d);
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
    return q8::launch_pdl(swiglu_quant_kernel, dim3(flat_grid(n4_total, 2)), dim3(kQuantThreads), 0,
                          static_cast<cudaStream_t>(stream), reinterpret_cast<const float4 *>(gate),
                          reinterpret_cast<const float4 *>(up), reinterpret_cast<float4 *>(y), n4_valid, n4_total,
                          reinterpret_cast<uint32_t *>(qs), ds);
}
