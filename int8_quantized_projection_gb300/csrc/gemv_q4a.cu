// gemv_q4a.cu -- batch-1 projection with asymmetric 4-bit weight blocks.
//
// y[i] = sum_b ( d(i,b) * d_a(b) * sum_e nib(i,b,e) * q_a(b,e)  -  m(i,b) * d_a(b) * ssum_a(b) )
//
// The block format and its dot product with a q8_0 activation chunk are in
// q4a_block.cuh.  Shapes whose activation fits the staged kernel of gemv.cu
// (k <= 65536) run there, instantiated for this format: per-warp rings fed by
// bulk copies, as for Q8_0 weights.  This file holds the path for longer rows:
// the activation (k bytes of codes + k/8 bytes of d|ssum) is staged once per
// CTA in shared memory, 144 bytes per 4-block chunk so that lanes reading
// different chunks hit different banks, and each lane streams its weight
// chunks from global memory with 16-byte loads.  Lanes per row = the next
// power of two of the row's chunk count (at most 32); warps take rows in a
// grid stride.
#include "q4a_block.cuh"

namespace {

using q8::kA4ChunkWords;
using q8::a4_chunk;

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
    if (nc <= q8::kGemvStagedMaxChunks)
        return q8::gemv_staged_q4a_launch(w, n, k, qs, ds, y, static_cast<cudaStream_t>(stream));
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

extern "C" int q4a_gemv_batched(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds,
                                int64_t tokens, float *y, void *stream)
{
    if (!w || !qs || !ds || !y || n < 1 || n > (int64_t(1) << 40) || k <= 0 || (k % 256) != 0 || tokens < 1 ||
        tokens > Q8_GEMV_MAX_TOKENS)
        return Q8_ERR_ARG;
    if (tokens == 1) return q4a_gemv(w, n, k, qs, ds, y, stream);
    if (!q8::aligned16(w) || !q8::aligned16(qs) || !q8::aligned16(ds) || !q8::aligned16(y)) return Q8_ERR_ALIGN;
    if (!q8::device_is_sm103()) return Q8_ERR_DEVICE;
    return q8::gemv_small_q4a_launch(w, n, k, qs, ds, y, tokens, static_cast<cudaStream_t>(stream));
}

extern "C" int q4a_gemv_batched_grouped(const q8_gemv_proj *projs, int count, int64_t k, const int8_t *qs,
                                        const uint32_t *ds, int64_t tokens, void *stream)
{
    if (!projs || count < 1 || count > Q8_MAX_GROUP || !qs || !ds || k <= 0 || (k % 256) != 0 || tokens < 1 ||
        tokens > Q8_GEMV_MAX_TOKENS)
        return Q8_ERR_ARG;
    for (int i = 0; i < count; ++i)
        if (!projs[i].w || !projs[i].y || projs[i].n < 1 || projs[i].n > (int64_t(1) << 40)) return Q8_ERR_ARG;
    if (!q8::aligned16(qs) || !q8::aligned16(ds)) return Q8_ERR_ALIGN;
    for (int i = 0; i < count; ++i)
        if (!q8::aligned16(projs[i].w) || !q8::aligned16(projs[i].y)) return Q8_ERR_ALIGN;
    if (!q8::device_is_sm103()) return Q8_ERR_DEVICE;
    if (tokens == 1) {  // one token: the batch-1 kernel, projection by projection (as q4a_gemv_batched)
        for (int i = 0; i < count; ++i) {
            const int st = q4a_gemv(projs[i].w, projs[i].n, k, qs, ds, projs[i].y, stream);
            if (st != Q8_OK) return st;
        }
        return Q8_OK;
    }
    return q8::gemv_small_q4a_grouped_launch(projs, count, k, qs, ds, tokens, static_cast<cudaStream_t>(stream));
}
