// gemv_q4a.cu -- batch-1 projection with asymmetric 4-bit weight blocks.
//
// y[i] = sum_b ( d(i,b) * d_a(b) * sum_e nib(i,b,e) * q_a(b,e)  -  m(i,b) * d_a(b) * ssum_a(b) )
//
// A weight block holds 32 values d * nib - m (f16 d, f16 m, unsigned 4-bit
// nib): the q4_K value form d*s*nib - dmin*m of "12 - r5-r6 re-ranking +
// structural rewrite spec" (sec. 3) with its two-level scales folded into one
// scale and one min per 32 elements.  Against a q8_0 activation block the min
// term needs no second dot product: m * d_a * sum_e q_e, and sum_e q_e is the
// int16 ssum that the plane carries for exactly this purpose ("54 - r51 -
// producer-fused A-quantize mode 1", sec. 2.1).
//
// Layout: a block is 20 bytes -- d at +0, m at +2, then byte j (j < 16) holds
// element j in its low nibble and element j + 16 in its high nibble -- so four
// blocks are 80 bytes = five 16-byte loads, and every block is five whole
// 32-bit words.  One nibble word gives two dp4a operands: w & 0x0f0f0f0f
// (elements 4i..4i+3) and (w >> 4) & 0x0f0f0f0f (elements 16+4i..16+4i+3).
// The activation (k bytes of codes + k/8 bytes of d|ssum) is staged once per
// CTA in shared memory, 144 bytes per 4-block chunk so that lanes reading
// different chunks hit different banks.  Lanes per row = the next power of two
// of the row's chunk count (at most 32); warps take rows in a grid stride.
#include "q8_common.cuh"

namespace {

constexpr int kA4ChunkWords = 20;   // 4 blocks x 5 words (80 bytes)
constexpr int kA4ActChunk = 144;    // 128 B codes + 16 B ds words
constexpr int kA4Threads = 256;

__device__ __forceinline__ uint4 ld_stream4(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Four blocks of one row (20 words) against the staged activation chunk.
__device__ __forceinline__ float a4_chunk(const uint32_t (&wv)[kA4ChunkWords], const uint8_t *ac, float acc)
{
    const uint4 dsv = *reinterpret_cast<const uint4 *>(ac + 128);
    const uint32_t dsw[4] = {dsv.x, dsv.y, dsv.z, dsv.w};
#pragma unroll
    for (int bb = 0; bb < 4; ++bb) {
        const uint4 a0 = *reinterpret_cast<const uint4 *>(ac + 32 * bb);
        const uint4 a1 = *reinterpret_cast<const uint4 *>(ac + 32 * bb + 16);
        const uint32_t aq[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        int isum = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t nw = wv[5 * bb + 1 + i];
            isum = q8::dp4a(nw & 0x0f0f0f0fu, aq[i], isum);             // elements 4i .. 4i+3
            isum = q8::dp4a((nw >> 4) & 0x0f0f0f0fu, aq[4 + i], isum);  // elements 16+4i .. 16+4i+3
        }
        const uint32_t dm = wv[5 * bb];
        const float dw = __half2float(__ushort_as_half(static_cast<unsigned short>(dm & 0xffffu)));
        const float mw = __half2float(__ushort_as_half(static_cast<unsigned short>(dm >> 16)));
        const float da = __half2float(__ushort_as_half(static_cast<unsigned short>(dsw[bb] & 0xffffu)));
        const int ssum = static_cast<int16_t>(static_cast<uint16_t>(dsw[bb] >> 16));
        // d*d_a and m*d_a are exact in f32 (11 + 11 significant bits)
        acc = __fmaf_rn(__fmul_rn(dw, da), static_cast<float>(isum), acc);
        acc = __fmaf_rn(-__fmul_rn(mw, da), static_cast<float>(ssum), acc);
    }
    return acc;
}

// Load chunks c and c + lpr of a row (zeros where invalid).
__device__ __forceinline__ void a4_load_pair(const uint4 *__restrict__ wr, int c, int lpr, bool v0, bool v1,
                                             uint32_t (&p0)[kA4ChunkWords], uint32_t (&p1)[kA4ChunkWords])
{
#pragma unroll
    for (int i = 0; i < 5; ++i) {
        const uint4 a = v0 ? ld_stream4(wr + c * 5 + i) : make_uint4(0u, 0u, 0u, 0u);
        const uint4 b = v1 ? ld_stream4(wr + (c + lpr) * 5 + i) : make_uint4(0u, 0u, 0u, 0u);
        p0[4 * i] = a.x; p0[4 * i + 1] = a.y; p0[4 * i + 2] = a.z; p0[4 * i + 3] = a.w;
        p1[4 * i] = b.x; p1[4 * i + 1] = b.y; p1[4 * i + 2] = b.z; p1[4 * i + 3] = b.w;
    }
}

__global__ void __launch_bounds__(kA4Threads)
q4a_gemv_kernel(const uint4 *__restrict__ w, int64_t n, int nc, const uint4 *__restrict__ qs,
                const uint4 *__restrict__ ds4, float *__restrict__ y, int lpr_log2)
{
    extern __shared__ __align__(16) uint8_t act[];
    const int lane = threadIdx.x & 31;
    const int lpr = 1 << lpr_log2, rpw = 32 >> lpr_log2;
    const int ri = lane >> lpr_log2, cj = lane & (lpr - 1);
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t groups = (n + rpw - 1) / rpw;
    const int64_t pitch4 = static_cast<int64_t>(nc) * 5;  // row pitch in 16-byte units
    const int nsteps = (nc + 2 * lpr - 1) / (2 * lpr);    // chunk pairs per row, the same for every lane

    // A warp walks (row group, step) items; each step is one pair of chunks
    // per lane, held in p0/p1 and loaded one item ahead.  The weights do not
    // depend on the previous kernel in the stream, so the first item is loaded
    // before waiting for it and before the activation is staged
    // (programmatic dependent launch).
    uint32_t p0[kA4ChunkWords], p1[kA4ChunkWords];
    auto load_item = [&](int64_t G, int step) {
        const int64_t row = G * rpw + ri;
        const int c = cj + 2 * lpr * step;
        const bool v0 = G < groups && row < n && c < nc;
        a4_load_pair(w + (v0 ? row : 0) * pitch4, c, lpr, v0, v0 && c + lpr < nc, p0, p1);
    };
    load_item(warp, 0);
    q8::griddep_launch_dependents();
    q8::griddep_wait();  // the plane may come from the previous kernel
    for (int idx = threadIdx.x; idx < nc * 9; idx += blockDim.x) {
        const int c = idx / 9, j = idx - c * 9;
        const uint4 v = (j < 8) ? __ldg(qs + c * 8 + j) : __ldg(ds4 + c);
        *reinterpret_cast<uint4 *>(act + c * kA4ActChunk + 16 * j) = v;
    }
    __syncthreads();

    float acc = 0.0f;
    int64_t G = warp;
    int step = 0;
    while (G < groups) {
        const int64_t row = G * rpw + ri;
        const int c = cj + 2 * lpr * step;
        if (row < n && c < nc) acc = a4_chunk(p0, act + c * kA4ActChunk, acc);
        if (row < n && c + lpr < nc) acc = a4_chunk(p1, act + (c + lpr) * kA4ActChunk, acc);
        int64_t Gn = G;
        int sn = step + 1;
        if (sn == nsteps) {
            sn = 0;
            Gn = G + nwarps;
        }
        load_item(Gn, sn);
        if (sn == 0) {  // row group complete: reduce over the lanes of each row
            for (int o = lpr >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(Q8_FULL_MASK, acc, o);
            if (cj == 0 && row < n) y[row] = acc;
            acc = 0.0f;
        }
        G = Gn;
        step = sn;
    }
}

int ceil_log2_a4(int v)
{
    int l = 0;
    while ((1 << l) < v) ++l;
    return l;
}

} // namespace

extern "C" int q4a_gemv(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, float *y,
                        void *stream)
{
    if (!w || !qs || !ds || !y || n < 1 || n > (int64_t(1) << 40) || k <= 0 || (k % 128) != 0) return Q8_ERR_ARG;
    if (!q8::aligned16(w) || !q8::aligned16(qs) || !q8::aligned16(ds) || !q8::aligned16(y)) return Q8_ERR_ALIGN;
    const int64_t nc = k / 128;
    const int64_t smem = nc * kA4ActChunk;
    if (smem > 227 * 1024) return Q8_ERR_ARG;  // the staged activation must fit in shared memory (k <= 206592)
    if (!q8::device_is_sm103()) return Q8_ERR_DEVICE;
    const int lpr_log2 = ceil_log2_a4(static_cast<int>(nc < 32 ? nc : 32));
    const int rpw = 32 >> lpr_log2;
    const int64_t groups = (n + rpw - 1) / rpw;
    const int sms = q8::device_sm_count();
    if (sms <= 0) return Q8_ERR_DEVICE;
    const int64_t warps_per_cta = kA4Threads / 32;
    int64_t grid = (groups + warps_per_cta - 1) / warps_per_cta;
    if (!q8::set_max_dynamic_smem(reinterpret_cast<const void *>(q4a_gemv_kernel), 227 * 1024, 5))
        return Q8_ERR_LAUNCH;
    // one wave of resident CTAs (each stages the activation once), warps walking rows in a grid stride
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, q4a_gemv_kernel, kA4Threads, static_cast<size_t>(smem)) !=
            cudaSuccess ||
        per_sm < 1)
        return Q8_ERR_LAUNCH;
    const int64_t cap = static_cast<int64_t>(sms) * per_sm;
    grid = grid < cap ? grid : cap;
    return q8::launch_pdl(q4a_gemv_kernel, dim3(static_cast<unsigned>(grid)), dim3(kA4Threads),
                          static_cast<size_t>(smem), static_cast<cudaStream_t>(stream), static_cast<const uint4 *>(w), n,
                          static_cast<int>(nc), reinterpret_cast<const uint4 *>(qs),
                          reinterpret_cast<const uint4 *>(ds), y, lpr_log2);
}
