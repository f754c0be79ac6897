// gemv.cu -- batch-1 Q8_0 x q8_0 projection (decode).
//
// y[i] = sum_b d_w(i,b) * d_a(b) * sum_j qw(i,b,j) * qa(b,j)
//
// The defects listed in "Part 4 - Lecture 05 - Fusion and the
// Activation-Quantization Discipline" (sec. 2.1-2.4) and how this kernel
// avoids them on GB300:
//   2.1  A 34-byte block is only 2-byte aligned.  Eight consecutive blocks
//        are 272 = 17 x 16 bytes, so when k/32 is a multiple of 8 every row
//        starts 16-byte aligned.  The weight stream is moved by cp.async.bulk
//        (the TMA unit) in pieces of up to 32 four-block chunks (136 bytes,
//        8-byte aligned) straight into shared memory; each lane reads its
//        chunk with conflict-free 8-byte shared loads (lanes 34 words apart)
//        and rebuilds the unaligned qs words with one byte-permute each.
//        Every warp owns a two-deep ring, and a CTA has up to 16 warps, so
//        an SM keeps ~139 KB of weights in flight and several warps per
//        scheduler to hide shared-memory latency.
//   2.2  The inner product is __dp4a on packed int8 words.
//   2.3  The activation (k bytes of qs + k/8 bytes of d|ssum) is staged once
//        per CTA in shared memory, 144 bytes per chunk so that lanes reading
//        different chunks hit different banks; no activation traffic reaches
//        HBM/L2 after the prologue.
//   2.4  Lanes per row is the next power of two of the row's chunk count
//        (capped at 32), so short rows share a warp instead of idling lanes;
//        the grid is a persistent set of at most one CTA per SM whose warp
//        count shrinks for small n, so small projections still spread over
//        many SMs.
// Two more modes of the same kernel (same weight stream, same per-row
// arithmetic, so the same output bits):
//   - fused producer (q8_0_gemv_fused): instead of copying a plane row, every
//     CTA computes the one-row producer (quantize, RMSNorm or SwiGLU) and its
//     q8_0 encoding straight into the staged activation, with the producer
//     arithmetic shared with the standalone kernels ("Part 4 - Lecture 05",
//     sec. 4: producer and consumer in one launch, one implementation);
//   - SwiGLU pairing (q8_0_gemv_gate_up): gate and up rows are interleaved in
//     units of 32 + 32 owned by one CTA, and the warp that completes a unit
//     writes the q8_0 block of silu(gate) * up, so the down projection's
//     plane comes out of this launch.
// Shapes whose k/32 is not a multiple of 8 (or whose activation would not
// fit in shared memory) use gemv_generic_kernel: plain 2-byte loads, the same
// lanes-per-row fitting, no staging.
#include <cooperative_groups.h>

#include "q4a_block.cuh"
#include "q8_common.cuh"

namespace cg = cooperative_groups;

namespace {

__device__ unsigned int g_gemv_err;

constexpr int kActChunkBytes = 144;             // 128 B qs + 16 B ds: 36 words, so lanes hit distinct banks
constexpr int kMaxActChunks = q8::kGemvStagedMaxChunks;  // k <= 65536 on the staged path

constexpr int kMaxProj = Q8_MAX_GROUP;        // projections of one activation per launch

struct GvProj {
    const uint8_t *w;  // n rows of Q8_0 blocks
    float *y;          // n outputs
    int64_t n;
    int64_t g_begin;   // first row group of this projection in the launch's group list
};

// Where the CTAs' staged activation comes from: a plane (row 0 of qs/ds),
// or one f32 row that every CTA encodes itself with the producer's own
// arithmetic (q8_0_gemv_fused).
struct GvAct {
    int producer;     // 0: plane; else Q8_PRODUCER_QUANT / _RMSNORM / _SWIGLU
    const float4 *a;  // x, or gate
    const float4 *b;  // up (SWIGLU)
    const float4 *w;  // RMSNorm weight
    float eps;
    int rms_j, rms_p; // the standalone RMSNorm's thread mapping for this k
};

// Geometry shared by all projections of a launch (they share k).
struct GvGeom {
    GvAct act;
    GvProj p[kMaxProj];
    int count;
    int nc;          // 4-block chunks per row (even: k/32 % 8 == 0)
    int lpr_log2;    // lanes per row = 1 << lpr_log2
    int rpw;         // rows per piece (1: a piece is up to 32*J chunks of one row)
    int ppr;         // pieces per row group
    int64_t groups;  // total row groups over all projections
    // SwiGLU pairing (q8_0_gemv_gate_up): projections 0 (gate) and 1 (up) of
    // equal n, one row per group.  Groups are interleaved in units of 32 gate
    // rows then the same 32 up rows, each CTA owns whole units, and the warp
    // that completes a unit writes the q8_0 block of silu(gate) * up.
    int pair_upc;       // 0: off; else the most units a CTA owns (sizes its buffer)
    int8_t *pair_qs;    // the SwiGLU output's plane row 0: n codes
    uint32_t *pair_ds;  // and its n/32 d|ssum words
};

// Shared bytes of the pairing buffer: per unit 64 f32 results and a counter.
__host__ __device__ inline int pair_region_bytes(int upc) { return upc ? (upc * (64 * 4 + 4) + 127) & ~127 : 0; }

// global row group -> projection index
__device__ __forceinline__ int proj_of(const GvGeom &g, int64_t G)
{
    int j = 0;
#pragma unroll
    for (int i = 1; i < kMaxProj; ++i)
        if (i < g.count && G >= g.p[i].g_begin) j = i;
    return j;
}

// global row group -> (projection, row group within it)
__device__ __forceinline__ void locate(const GvGeom &g, int64_t G, int &pi, int64_t &Gl)
{
    if (g.pair_upc) {
        const int w = static_cast<int>(G & 63);
        pi = w >> 5;
        Gl = (G >> 6) * 32 + (w & 31);
        return;
    }
    pi = proj_of(g, G);
    Gl = G - g.p[pi].g_begin;
}

// A weight format of the staged kernel: the bytes of four consecutive blocks
// of a row (a "chunk", k = 128), how many chunks a lane takes per ring slot
// (J), the ring depth per warp, the warps per CTA, and the chunk's dot product
// with a staged activation chunk (128 B of codes + 4 d|ssum words).  A ring
// slot ("piece") holds 32*J chunks: up to 32*J chunks of one row, or whole
// rows when a row has at most 32 chunks.
//
// Q8_0: a chunk is 136 bytes, 8-byte aligned in shared memory when rows start
// 16-byte aligned (k/32 % 8 == 0); lanes read 8 bytes at a time, 34 words
// apart, so a half-warp touches 32 distinct banks.
#ifndef Q8_Q80_STAGES
#define Q8_Q80_STAGES 2
#endif
#ifndef Q8_Q80_J
#define Q8_Q80_J 1
#endif
#ifndef Q8_Q80_WARPS
#define Q8_Q80_WARPS 16
#endif
struct FmtQ8_0 {
    static constexpr bool kFused = true;  // produced rows (q8_0_gemv_fused) and gate/up pairing (q8_0_gemv_gate_up)
    static constexpr int kChunkBytes = 136;
    static constexpr int kLaneChunks = Q8_Q80_J;
    static constexpr int kStages = Q8_Q80_STAGES;
    static constexpr int kWarps = Q8_Q80_WARPS;
    __device__ static float dot(const uint8_t *wc, const uint8_t *ac);
};

// Asymmetric 4-bit blocks (q4a_block.cuh): a chunk is 80 bytes, 16-byte
// aligned; lanes read it as five 16-byte words, 20 words apart, so each
// quarter-warp touches 32 distinct banks.  At 80 bytes per 128 elements the
// same HBM rate needs 1.7x the chunk rate of Q8_0, and the kernel is bound by
// the latency of each warp's chunk arithmetic, so this format runs more
// independent chunks at once (more warps, or more chunks per lane).
#ifndef Q8_Q4A_STAGES
#define Q8_Q4A_STAGES 2
#endif
#ifndef Q8_Q4A_J
#define Q8_Q4A_J 2
#endif
#ifndef Q8_Q4A_WARPS
#define Q8_Q4A_WARPS 16
#endif
struct FmtQ4A {
    static constexpr bool kFused = false;  // plane input and y outputs only
    static constexpr int kChunkBytes = q8::kA4ChunkBytes;
    static constexpr int kLaneChunks = Q8_Q4A_J;
    static constexpr int kStages = Q8_Q4A_STAGES;
    static constexpr int kWarps = Q8_Q4A_WARPS;
    __device__ static float dot(const uint8_t *wc, const uint8_t *ac)
    {
        uint32_t wv[q8::kA4ChunkWords];
#pragma unroll
        for (int c = 0; c < 5; ++c) {
            const uint4 v = *reinterpret_cast<const uint4 *>(wc + 16 * c);
            wv[4 * c + 0] = v.x;
            wv[4 * c + 1] = v.y;
            wv[4 * c + 2] = v.z;
            wv[4 * c + 3] = v.w;
        }
        return q8::a4_chunk(wv, ac, 0.0f);
    }
};

// header: per-warp mbarriers, per-warp stage metadata, the CTA's row-group counter
template <class F>
__host__ __device__ inline int smem_header_bytes() { return F::kWarps * F::kStages * 8 * 2 + 128; }

// One 4-block Q8_0 chunk: 34 words of raw weights (shared memory, 8-byte
// aligned) against 128 B of qs and 4 ds words of the activation.
__device__ __forceinline__ float FmtQ8_0::dot(const uint8_t *wc, const uint8_t *ac)
{
    uint32_t wv[34];
#pragma unroll
    for (int c = 0; c < 17; ++c) {
        const uint2 v = *reinterpret_cast<const uint2 *>(wc + 8 * c);
        wv[2 * c + 0] = v.x;
        wv[2 * c + 1] = v.y;
    }
    const uint4 ad = *reinterpret_cast<const uint4 *>(ac + 128);
    const uint32_t adw[4] = {ad.x, ad.y, ad.z, ad.w};
    float acc = 0.0f;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const uint4 a0 = *reinterpret_cast<const uint4 *>(ac + 32 * b);
        const uint4 a1 = *reinterpret_cast<const uint4 *>(ac + 32 * b + 16);
        const uint32_t aq[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        // block b: f16 d at byte 34b, qs at 34b + 2 (word-aligned for odd b only)
        const uint32_t dbits = (b & 1) ? (wv[(17 * b - 1) / 2] >> 16) : (wv[17 * b / 2] & 0xffffu);
        int isum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int o = 34 * b + 2 + 4 * i;
            const uint32_t qw = (o & 3) ? __byte_perm(wv[o >> 2], wv[(o >> 2) + 1], 0x5432) : wv[o >> 2];
            isum = q8::dp4a(qw, aq[i], isum);
        }
        const float dw = __half2float(__ushort_as_half(static_cast<unsigned short>(dbits)));
        const float da = __half2float(__ushort_as_half(static_cast<unsigned short>(adw[b] & 0xffffu)));
        acc = fmaf(dw * da, static_cast<float>(isum), acc);  // dw*da is exact in f32
    }
    return acc;
}

// Fused activation staging: the producer's f32 row and its q8_0 encoding,
// computed by this CTA into the staged layout (chunk c: 32 qs words, then
// the d|ssum words of its 4 blocks).  A pair of adjacent threads encodes one
// 32-element block (pair i takes blocks i, i + blockDim.x/2, ...; thread half
// h holds elements 16h..16h+15): the block's amax and code sum are register
// reductions and one shuffle, and d and 1/d are computed once per thread
// (the codes are those any other split of the block gives: a maximum,
// elementwise codes and an integer sum).  Every input of a thread's first
// block (x and the norm weight, or gate and up) is loaded before anything
// else, so for RMSNorm those loads are in flight together with the loads of
// the sum of squares: the prologue waits for one round trip to L2.  The
// row's sum of squares is formed exactly as the standalone kernel forms it
// with P threads: this CTA's warps play its P/32 warps in turn (a CTA's
// thread count is a multiple of 32, so lane l plays lane l), `red` collects
// the warp sums, and every thread adds them in warp order.
__device__ __forceinline__ void stage_produced(const GvGeom &g, uint8_t *act, float *red, int warp, int lane)
{
    constexpr int kBatch = 4;  // loads a thread keeps in flight before it uses them
    const int nwarps = static_cast<int>(blockDim.x >> 5);
    const int nblk = g.nc * 4;  // 32-element blocks of the row
    const int F = g.nc * 32;    // float4 per row
    const GvAct &A = g.act;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    const bool second = A.producer != Q8_PRODUCER_QUANT;  // norm weight (RMSNorm) or up (SwiGLU)
    const float4 *pa = A.a;
    const float4 *pb = A.producer == Q8_PRODUCER_SWIGLU ? A.b : A.w;
    const int h = lane & 1;                                   // half of the block
    const int pstride = static_cast<int>(blockDim.x >> 1);    // thread pairs
    int blk = static_cast<int>(threadIdx.x >> 1);
    float4 va[4], vb[4];
    auto load = [&](int b) {
#pragma unroll
        for (int e = 0; e < 4; ++e) va[e] = __ldg(pa + 8 * b + 4 * h + e);
        if (second)
#pragma unroll
            for (int e = 0; e < 4; ++e) vb[e] = __ldg(pb + 8 * b + 4 * h + e);
    };
    if (blk < nblk) load(blk);
    float scale = 0.0f;
    if (A.producer == Q8_PRODUCER_RMSNORM) {
        const int vws = A.rms_p >> 5;
        for (int vw = warp; vw < vws; vw += nwarps) {
            const int vt = vw * 32 + lane;
            float ss = 0.0f;
            for (int j0 = 0; j0 < A.rms_j; j0 += kBatch) {
                float4 v[kBatch];
#pragma unroll
                for (int u = 0; u < kBatch; ++u) {
                    const int f = vt + (j0 + u) * A.rms_p;
                    v[u] = (j0 + u < A.rms_j && f < F) ? __ldg(pa + f) : zero;
                }
#pragma unroll
                for (int u = 0; u < kBatch; ++u) ss = q8::rms_sumsq4(ss, v[u]);  // zeros leave ss as it is
            }
            ss = q8::rms_warp_sum(ss);
            if (lane == 0) red[vw] = ss;
        }
        __syncthreads();
        float tot = 0.0f;
        for (int i = 0; i < vws; ++i) tot += red[i];
        scale = q8::rms_scale(tot, F * 4, A.eps);
    }
    // the pairs stay whole through the loop: blockDim.x is even and the pair's
    // threads see the same block index, so both take part in every shuffle
    for (int first = 1; blk < nblk; blk += pstride, first = 0) {
        if (!first) load(blk);  // a later block (rows longer than 16 x threads)
        float amax = 0.0f;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float4 o = va[e];
            if (A.producer == Q8_PRODUCER_RMSNORM)
                o = q8::rms_apply4(o, scale, vb[e]);
            else if (A.producer == Q8_PRODUCER_SWIGLU)
                o = q8::silu_mul4(o, vb[e]);
            va[e] = o;
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(o.x), fabsf(o.y)), fmaxf(fabsf(o.z), fabsf(o.w))));
        }
        const unsigned pair_mask = 3u << (lane & ~1);
        amax = fmaxf(amax, __shfl_xor_sync(pair_mask, amax, 1));
        const float d = q8::q8_block_d(amax);
        const float di = q8::q8_block_di(d);
        uint32_t qw[4];
        int sum = 0;
        if (q8::block_rounds_by_add(d)) {  // codes rounded on the FMA pipe (q8_common.cuh)
            uint32_t bsum = 0u;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                uint32_t b0, b1, b2, b3;
                q8::round_by_add2(va[e].x, va[e].y, di, b0, b1);
                q8::round_by_add2(va[e].z, va[e].w, di, b2, b3);
                bsum += b0 + b1 + b2 + b3;
                qw[e] = __byte_perm(__byte_perm(b0, b1, 0x0040u), __byte_perm(b2, b3, 0x0040u), 0x5410u);
            }
            sum = static_cast<int>(bsum - 16u * q8::kRoundMagicBits);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c0 = q8::q8_code(va[e].x, di), c1 = q8::q8_code(va[e].y, di);
                const int c2 = q8::q8_code(va[e].z, di), c3 = q8::q8_code(va[e].w, di);
                sum += c0 + c1 + c2 + c3;
                qw[e] = q8::pack4(c0, c1, c2, c3);
            }
        }
        sum += __shfl_xor_sync(pair_mask, sum, 1);
        uint8_t *ch = act + (blk >> 2) * kActChunkBytes;
        *reinterpret_cast<uint4 *>(ch + 32 * (blk & 3) + 16 * h) = make_uint4(qw[0], qw[1], qw[2], qw[3]);
        if (h == 0) reinterpret_cast<uint32_t *>(ch + 128)[blk & 3] = q8::q8_dsword(d, sum);
    }
}

template <class F>
__global__ void __launch_bounds__(F::kWarps * 32)
gemv_staged_kernel(const uint4 *__restrict__ qs_row, const uint32_t *__restrict__ ds_row,
                   const __grid_constant__ GvGeom g)
{
    constexpr int kChunkBytes = F::kChunkBytes;
    constexpr int J = F::kLaneChunks;
    constexpr int kStages = F::kStages;
    constexpr int kWarps = F::kWarps;
    constexpr int kPieceChunks = 32 * J;
    constexpr int kPieceBytes = kPieceChunks * kChunkBytes;  // a multiple of 16 bytes
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem);
    int2 *meta = reinterpret_cast<int2 *>(smem + kWarps * kStages * 8);  // (row group, piece) per stage
    unsigned int *counter = reinterpret_cast<unsigned int *>(smem + kWarps * kStages * 16);
    uint8_t *act = smem + smem_header_bytes<F>();
    uint8_t *pairs = act + ((g.nc * kActChunkBytes + 127) & ~127);
    float *pbuf = reinterpret_cast<float *>(pairs);                                 // [unit][64]
    unsigned int *pcnt = reinterpret_cast<unsigned int *>(pbuf + 64 * g.pair_upc);  // [unit]
    uint8_t *ring = pairs + pair_region_bytes(g.pair_upc);
    uint64_t *mybar = bars + warp * kStages;
    int2 *mymeta = meta + warp * kStages;
    uint8_t *myring = ring + warp * kStages * kPieceBytes;

    // This CTA owns a contiguous range of row groups; its warps take groups
    // from it one at a time (a warp always computes whole rows, so the result
    // does not depend on which warp takes which group).
    const int64_t pitch = static_cast<int64_t>(g.nc) * kChunkBytes;
    int64_t cg0 = g.groups * blockIdx.x / gridDim.x;
    int64_t cg1 = g.groups * (blockIdx.x + 1) / gridDim.x;
    if (g.pair_upc) {  // whole units of 64 groups
        const int64_t units = g.groups >> 6;
        cg0 = (units * blockIdx.x / gridDim.x) << 6;
        cg1 = (units * (blockIdx.x + 1) / gridDim.x) << 6;
    }
    const unsigned int ngroups = static_cast<unsigned int>(cg1 - cg0);

    // lane 0's fetch cursor
    int fetch_grp = -1, fetch_p = 0;
    bool fetch_done = false;
    auto issue = [&](int s) {
        int grp = -1, p = 0;
        if (!fetch_done) {
            if (fetch_grp >= 0 && fetch_p < g.ppr) {
                grp = fetch_grp;
                p = fetch_p++;
            } else {
                const unsigned int gn = atomicAdd(counter, 1u);
                if (gn < ngroups) {
                    fetch_grp = grp = static_cast<int>(gn);
                    fetch_p = 1;
                    p = 0;
                } else {
                    fetch_done = true;
                }
            }
        }
        mymeta[s] = make_int2(grp, p);
        if (grp < 0) {  // nothing left: complete the phase so the warp sees the end marker
            q8::mbar_arrive(&mybar[s]);
            return;
        }
        const int64_t G = cg0 + grp;
        int pi;
        int64_t Gl;  // row group within the projection
        locate(g, G, pi, Gl);
        const GvProj &pj = g.p[pi];
        const uint8_t *src;
        uint32_t bytes;
        if (g.rpw == 1) {  // one row per piece, up to 32*J chunks of it
            const int chunks = min(kPieceChunks, g.nc - kPieceChunks * p);
            bytes = static_cast<uint32_t>(chunks * kChunkBytes);
            src = pj.w + Gl * pitch + static_cast<int64_t>(kPieceChunks) * p * kChunkBytes;
        } else {
            const int64_t r0 = Gl * g.rpw;
            const int64_t rows = min(static_cast<int64_t>(g.rpw), pj.n - r0);
            bytes = static_cast<uint32_t>(rows * pitch);
            src = pj.w + r0 * pitch;
        }
        q8::mbar_arrive_expect_tx(&mybar[s], bytes);
        q8::bulk_g2s(myring + s * kPieceBytes, src, bytes, &mybar[s]);
    };

    if (threadIdx.x == 0) *counter = 0u;
    for (int i = threadIdx.x; i < g.pair_upc; i += blockDim.x) pcnt[i] = 0u;
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) q8::mbar_init(&mybar[s], 1);
        q8::fence_mbar_init();
    }
    __syncthreads();
    // The weights do not depend on the previous kernel in the stream: start
    // streaming them before waiting for it (programmatic dependent launch).
    if (lane == 0)
        for (int s = 0; s < kStages; ++s) issue(s);
    if (g.act.producer == Q8_PRODUCER_RMSNORM)  // the norm weight is a constant input too: to L1 now
        for (int l = threadIdx.x; l < g.nc * 4; l += blockDim.x)  // 128-byte lines of k floats
            asm volatile("prefetch.global.L1 [%0];" ::"l"(g.act.w + 8 * l));
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (g.act.producer == 0) {
        // stage the activation: chunk c = 8 x 16 B of qs then its 4 ds words
        for (int idx = threadIdx.x; idx < g.nc * 9; idx += blockDim.x) {
            const int c = idx / 9, j = idx - c * 9;
            const uint4 v = (j < 8) ? __ldg(qs_row + c * 8 + j) : __ldg(reinterpret_cast<const uint4 *>(ds_row) + c);
            *reinterpret_cast<uint4 *>(act + c * kActChunkBytes + 16 * j) = v;
        }
    } else if constexpr (F::kFused) {
        // RMSNorm's warp sums: the free upper 64 bytes of the header's last 128
        stage_produced(g, act, reinterpret_cast<float *>(counter + 16), warp, lane);
    }
    __syncthreads();

    // Lane roles.  Long rows (rpw == 1): slot j of a piece is chunk
    // 32*J*p + 32*j + lane of the row.  Short rows: lanes (ri, cj) with
    // 1 << lpr_log2 lanes per row; slot j is row j*(32 >> lpr_log2) + ri of the
    // piece, chunk cj.
    const int lpr = 1 << g.lpr_log2;
    const int rps = 32 >> g.lpr_log2;          // rows per slot
    const int ri = lane >> g.lpr_log2;         // row within a slot
    const int cj = lane & (lpr - 1);           // chunk within a row
    float acc[J];
#pragma unroll
    for (int j = 0; j < J; ++j) acc[j] = 0.0f;
    for (uint32_t i = 0;; ++i) {
        const int s = static_cast<int>(i % kStages);
        const uint32_t par = (i / kStages) & 1u;
        const bool ok = q8::mbar_wait_bounded(&mybar[s], par);
        if (!__all_sync(Q8_FULL_MASK, ok)) {
            if (lane == 0) atomicOr(&g_gemv_err, 1u);
            // before leaving, let this warp's copies in flight land (each
            // wait bounded): no copy may still write into shared memory once
            // the CTA has exited
            for (uint32_t j = 0; j < static_cast<uint32_t>(kStages); ++j)
                (void)q8::mbar_wait_bounded(&mybar[(i + j) % kStages], ((i + j) / kStages) & 1u, Q8_DRAIN_LIMIT_NS);
            return;
        }
        const int2 m = mymeta[s];
        if (m.x < 0) break;
        const uint8_t *buf = myring + s * kPieceBytes;
        const int64_t G = cg0 + m.x;
        int pi;
        int64_t Gl;
        locate(g, G, pi, Gl);
        const GvProj &pj = g.p[pi];
        const int p = m.y;
#pragma unroll
        for (int j = 0; j < J; ++j) {
            int chunk, soff;
            bool valid;
            if (g.rpw == 1) {
                chunk = kPieceChunks * p + 32 * j + lane;
                soff = (32 * j + lane) * kChunkBytes;
                valid = chunk < g.nc;
            } else {
                const int rr = j * rps + ri;  // row within the piece
                chunk = cj;
                soff = (rr * g.nc + cj) * kChunkBytes;
                valid = cj < g.nc && Gl * g.rpw + rr < pj.n;
            }
            if (valid) acc[j] += F::dot(buf + soff, act + chunk * kActChunkBytes);
        }
        __syncwarp();
        if (lane == 0) issue(s);  // refill the slot just consumed
        if (p == g.ppr - 1) {     // row group complete: reduce over the lanes of each row
            if (g.rpw == 1) {
                float a = acc[0];
#pragma unroll
                for (int j = 1; j < J; ++j) a += acc[j];
                for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(Q8_FULL_MASK, a, o);
                if (lane == 0 && pj.y) pj.y[Gl] = a;  // y may be absent only in pairing mode
                if (F::kFused && g.pair_upc) {
                    // this row's result into its unit; the warp that brings the
                    // unit's count to 64 encodes silu(gate) * up for its 32 rows
                    const int64_t ul = m.x >> 6;  // unit within this CTA (cg0 is unit-aligned)
                    const int w = static_cast<int>(G & 63);
                    unsigned int done = 0u;
                    if (lane == 0) {
                        pbuf[ul * 64 + w] = a;
                        __threadfence_block();            // release this row's value
                        done = atomicAdd(&pcnt[ul], 1u);
                        __threadfence_block();            // acquire the other rows' values
                    }
                    done = __shfl_sync(Q8_FULL_MASK, done, 0);
                    if (done == 63u) {
                        __syncwarp();  // orders lane 0's acquire before every lane's reads
                        const float gv = pbuf[ul * 64 + lane], uv = pbuf[ul * 64 + 32 + lane];
                        uint32_t dsw;
                        const int q = q8::q8_encode32(q8::silu_mul(gv, uv), dsw);
                        const int64_t unit = G >> 6;
                        g.pair_qs[unit * 32 + lane] = static_cast<int8_t>(q);
                        if (lane == 0) g.pair_ds[unit] = dsw;
                    }
                }
            } else {
#pragma unroll
                for (int j = 0; j < J; ++j) {
                    float a = acc[j];
                    for (int o = lpr >> 1; o > 0; o >>= 1) a += __shfl_xor_sync(Q8_FULL_MASK, a, o);
                    const int64_t row = Gl * g.rpw + j * rps + ri;
                    if (cj == 0 && row < pj.n) pj.y[row] = a;
                }
            }
#pragma unroll
            for (int j = 0; j < J; ++j) acc[j] = 0.0f;
        }
    }
}

// Generic path: any k % 32 == 0.  Warp = 32 / lpr rows; lane (i, j) handles
// blocks j, j + lpr, ... of row r0 + i.  blockIdx.y selects the token (the
// same kernel serves the GEMM's odd shapes).
__global__ void __launch_bounds__(128)
gemv_generic_kernel(const uint8_t *__restrict__ w, int64_t n, int nb, const int8_t *__restrict__ qs,
                    const uint32_t *__restrict__ ds, float *__restrict__ y, int lpr_log2)
{
    q8::griddep_launch_dependents();
    q8::griddep_wait();  // the plane may come from the previous kernel
    const int lane = threadIdx.x & 31;
    const int lpr = 1 << lpr_log2;
    const int rpw = 32 >> lpr_log2;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t tok = blockIdx.y;
    const int64_t row = warp * rpw + (lane >> lpr_log2);
    const int j = lane & (lpr - 1);
    const int64_t pitch = static_cast<int64_t>(nb) * 34;
    const int8_t *qa = qs + tok * static_cast<int64_t>(nb) * 32;
    const uint32_t *da = ds + tok * nb;
    float acc = 0.0f;
    if (row < n) {
        const uint16_t *wr = reinterpret_cast<const uint16_t *>(w + row * pitch);
        for (int b = j; b < nb; b += lpr) {
            const uint16_t *blk = wr + 17 * b;
            const uint4 a0 = __ldg(reinterpret_cast<const uint4 *>(qa + 32 * b));
            const uint4 a1 = __ldg(reinterpret_cast<const uint4 *>(qa + 32 * b + 16));
            const uint32_t aq[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            int isum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t qw = static_cast<uint32_t>(__ldg(blk + 1 + 2 * i)) |
                                    (static_cast<uint32_t>(__ldg(blk + 2 + 2 * i)) << 16);
                isum = q8::dp4a(qw, aq[i], isum);
            }
            const float dw = __half2float(__ushort_as_half(__ldg(blk)));
            const float dav = __half2float(__ushort_as_half(static_cast<unsigned short>(__ldg(da + b) & 0xffffu)));
            acc = fmaf(dw * dav, static_cast<float>(isum), acc);
        }
    }
    for (int o = lpr >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(Q8_FULL_MASK, acc, o);
    if (j == 0 && row < n) y[tok * n + row] = acc;
}

// ---------------------------------------------------------------------------
// Small-batch path: t = 1..16 tokens against one weight matrix, the weights
// streamed from HBM once for all tokens (a decode step batched over a few
// sequences; the bridge between the batch-1 GEMV and the prefill GEMM).
// dp4a would need 8*t integer instructions per 4-byte weight word, more than
// an SM issues at HBM rate for t = 16, so the block dot products run on the
// tensor cores: mma.sync m16n8k16 on the int8 codes widened exactly to f16,
// two MMAs per 32-wide block and 8 tokens, whose f32 result is the exact
// integer dot product (|isum| <= 32*127*127 < 2^24).  (The int8 mma.sync
// needs no widening but its rate on this GPU falls short of HBM at t = 16.)
// Within a block the k order is permuted so that thread t4 of a quad holds
// code words t4 and t4 + 4 of the block (the integer sum does not depend on
// the order, and A and B use the same one); with rows 68 words apart in shared
// memory the 32 lanes of a warp then read 32 distinct banks.  Per block the
// scale is applied as in the GEMM: acc += (d_w * d_a) * isum.
//
// Work split: a CTA computes kSbRows weight rows for all tokens over a slice
// of k, in stages of kSbPieces "pieces" of 8 blocks (272 bytes of each row,
// contiguous in memory, so a stage reads kSbPieces*272 consecutive bytes per
// row).  One thread of a ninth warp moves each stage with three TMA loads:
// the weights (one 3-D box: rows x pieces x 272 bytes), the tokens' code
// bytes (128-byte boxes, 128-byte swizzled so fragment reads spread over the
// banks) and their d|ssum words; rows past n and tokens past t arrive as
// zeros.  Consumer warp w takes 16 rows (tile w % (kSbRows/16)) and one piece
// (w / (kSbRows/16)) of every stage.  For more than 8 tokens the consumer
// warps first widen the stage's activation codes to f16 together, in the
// order of the MMA's B fragments, and unpack its scales (sb_prep_act).  The
// CTAs of a thread-block cluster (1..8) split k between them, so narrow
// matrices still fill the GPU; one launch may cover several projections of
// the same activation (their row tiles form one grid).  Partial sums are
// added in piece order inside a CTA, then in cluster-rank order (every CTA
// finishes a share of the outputs, reading its peers' shared memory):
// results are run-to-run identical.
// ---------------------------------------------------------------------------
#ifndef Q8_SB_PIECES
#define Q8_SB_PIECES 1
#endif
#ifndef Q8_SB_S8_TILES
#define Q8_SB_S8_TILES 1  // token tiles up to which the block step runs on the int8 MMA
#endif
#ifndef Q8_SB_STAGES
#define Q8_SB_STAGES 2
#endif
#ifndef Q8_SB_WARPS
#define Q8_SB_WARPS 8
#endif
constexpr int kSbWarps = Q8_SB_WARPS;                    // consumer warps
constexpr int kSbThreads = (kSbWarps + 1) * 32;          // + the producer warp
constexpr int kSbPieces = Q8_SB_PIECES;                  // 8-block pieces per row and stage (1, 2 or 4)
constexpr int kSbRows = 16 * kSbWarps / kSbPieces;       // weight rows per CTA
constexpr int kSbTiles = kSbRows / 16;                   // 16-row MMA tiles per CTA
constexpr int kSbGroup = 8;                              // weight blocks per piece
constexpr int kSbMaxTokens = 16;
// stage layout (offsets from a 1024-byte aligned stage base); the weight part
// depends on the block format (SbLayout below)
constexpr int kSbOffAct = 0;                             // 2*kSbPieces boxes x 16 tokens x 128 B, swizzled
constexpr int kSbOffDs = kSbPieces * 4096;               // 16 tokens x 8*kSbPieces words
constexpr int kSbOffW = kSbOffDs + kSbPieces * 512;      // kSbRows rows x the format's row bytes
constexpr int kSbStages = Q8_SB_STAGES;
constexpr int kSbMaxCluster = 8;
static_assert(kSbPieces == 1 || kSbPieces == 2 || kSbPieces == 4, "pieces per stage");
static_assert(kSbStages * 16 + 8 <= 128, "barrier area");
static_assert(kSbOffW % 128 == 0, "TMA destination alignment");

// Weight block formats of the small-batch kernel.  codes<BB>(row, t4) returns
// the two 4-code words of block BB that thread t4 of a quad feeds the MMA (the
// block's elements 4*t4.. and 16 + 4*t4.., matching the activation's words t4
// and t4 + 4); d<BB> and m<BB> its scale and min.
struct SbQ8_0 {  // 34-byte blocks: f16 d, 32 int8 codes
    static constexpr int kBlockBytes = 34;
    static constexpr bool kMin = false;
    template <int BB>
    __device__ static uint2 codes(const uint8_t *row, int t4)
    {
        constexpr int off = 34 * BB + 2;  // the codes of block BB (row pieces start 16-byte aligned)
        if constexpr ((off & 3) == 0) {
            const uint32_t *p = reinterpret_cast<const uint32_t *>(row + off);
            return make_uint2(p[t4], p[t4 + 4]);
        } else {
            const uint32_t *p = reinterpret_cast<const uint32_t *>(row + off - 2);
            return make_uint2(__byte_perm(p[t4], p[t4 + 1], 0x5432), __byte_perm(p[t4 + 4], p[t4 + 5], 0x5432));
        }
    }
    template <int BB>
    __device__ static float d(const uint8_t *row)
    {
        return __half2float(*reinterpret_cast<const __half *>(row + 34 * BB));
    }
    template <int BB>
    __device__ static float m(const uint8_t *)
    {
        return 0.0f;
    }
};

// Asymmetric 4-bit blocks (q4a_block.cuh): 20 bytes, f16 d, f16 m, then byte j
// holding element j (low nibble) and element j + 16 (high nibble).  Nibble
// word t4 is exactly the thread's pair: its low nibbles are elements
// 4*t4.. and its high nibbles elements 16 + 4*t4.., as unsigned bytes 0..15.
struct SbQ4A {
    static constexpr int kBlockBytes = q8::kA4ChunkBytes / 4;
    static constexpr bool kMin = true;
    template <int BB>
    __device__ static uint2 codes(const uint8_t *row, int t4)
    {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(row + 20 * BB + 4 + 4 * t4);
        return make_uint2(w & 0x0f0f0f0fu, (w >> 4) & 0x0f0f0f0fu);
    }
    template <int BB>
    __device__ static float d(const uint8_t *row)
    {
        return __half2float(*reinterpret_cast<const __half *>(row + 20 * BB));
    }
    template <int BB>
    __device__ static float m(const uint8_t *row)
    {
        return __half2float(*reinterpret_cast<const __half *>(row + 20 * BB + 2));
    }
};

template <class W>
struct SbLayout {
    static constexpr int kPieceBytes = kSbGroup * W::kBlockBytes;   // 272 (Q8_0), 160 (Q4A): multiples of 16
    static constexpr int kRowBytes = kSbPieces * kPieceBytes;       // weight bytes per row and stage
    static constexpr int kStageTx = kSbOffW + kSbRows * kRowBytes;  // bytes the TMA writes per stage
    // the f16 path's prepared activation (written by the consumer warps, not
    // the TMA): codes as f16 in fragment order [block][token][t4][4 words],
    // and per (block, token tile, t4) {d_a, d_a, ssum, ssum} of tokens
    // 8j + 2*t4 and 8j + 2*t4 + 1 as f32
    static constexpr int kOffAh = (kStageTx + 127) / 128 * 128;
    static constexpr int kOffDc = kOffAh + kSbPieces * kSbGroup * kSbMaxTokens * 64;
    static constexpr int kStageBytes = (kOffDc + kSbPieces * kSbGroup * 2 * 4 * 16 + 1023) / 1024 * 1024;
    static constexpr int kOffBar = kSbStages * kStageBytes;         // full[], empty[], error flag
    static constexpr int kSmem = kOffBar + 128 + 1024;              // + alignment slack
    static_assert(kPieceBytes % 16 == 0, "TMA box rows");
    static_assert(kSbMaxTokens * kSbRows * kSbPieces * 4 <= kSbStages * kStageBytes, "partial sums reuse the ring");
};

__device__ __forceinline__ void mma_f16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Code words t4 and t4 + 4 of block BB of token tok in the stage's activation
// boxes: box 2*pc + BB/4, 16-byte chunks 2*(BB%4) and 2*(BB%4) + 1 of the
// token's 128-byte line, XOR-swizzled by tok % 8.
template <int BB>
__device__ __forceinline__ uint2 sb_act(const uint8_t *stage, int pc, int tok, int t4)
{
    constexpr int c0 = 2 * (BB & 3);
    const uint8_t *line = stage + kSbOffAct + (2 * pc + (BB >> 2)) * 2048 + tok * 128;
    return make_uint2(*reinterpret_cast<const uint32_t *>(line + ((c0 ^ (tok & 7)) << 4) + 4 * t4),
                      *reinterpret_cast<const uint32_t *>(line + (((c0 + 1) ^ (tok & 7)) << 4) + 4 * t4));
}

// Per output and block: acc += (d_w * d_a) * P, the scale rounded once, then
// for asymmetric weights acc += (-(m * d_a)) * ssum (both products exact in
// f32), packed in token pairs.  P is the exact integer block dot.
template <class W>
__device__ __forceinline__ void sb_epilogue(float2 (&acc)[2], const float (&c)[4], float dlo, float dhi, float mlo,
                                            float mhi, float2 da, float2 ss)
{
    acc[0] = __ffma2_rn(__fmul2_rn(make_float2(dlo, dlo), da), make_float2(c[0], c[1]), acc[0]);
    acc[1] = __ffma2_rn(__fmul2_rn(make_float2(dhi, dhi), da), make_float2(c[2], c[3]), acc[1]);
    if constexpr (W::kMin) {
        acc[0] = __ffma2_rn(__fmul2_rn(make_float2(-mlo, -mlo), da), ss, acc[0]);
        acc[1] = __ffma2_rn(__fmul2_rn(make_float2(-mhi, -mhi), da), ss, acc[1]);
    }
}

// One 32-wide block (block BB of piece `pc` of the stage) for this warp's 16
// rows (row g's piece at wpiece) and NT groups of 8 tokens (tokens past t
// are zeros), on the f16 MMA with the codes widened exactly.  Thread
// (g = lane/4, t4 = lane%4) holds the MMA fragments of rows g, g+8 and token
// g (+8 per token tile); its results are rows g, g+8 at tokens 2*t4, 2*t4+1
// (+8 per token tile), kept as token pairs.  da[j] is the d_a pair of tile j.
template <class W, int BB, int NT>
__device__ __forceinline__ void sb_block(const uint8_t *wpiece, const uint8_t *stage, int pc, int g, int t4,
                                         float2 (&acc)[NT][2])
{
    using L = SbLayout<W>;
    constexpr int kRowBytes = L::kRowBytes;
    const int bb = pc * kSbGroup + BB;  // block of the stage
    uint32_t bf[NT][4];  // token 8j+g: step 0 {codes 0,1 | 2,3} of word t4, step 1 the same of word t4 + 4
    float2 da[NT], ss[NT];  // d_a and ssum of tokens 8j + 2*t4, 8j + 2*t4 + 1
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const uint4 v = *reinterpret_cast<const uint4 *>(stage + L::kOffAh + (((bb * kSbMaxTokens + 8 * j + g) * 4 + t4)
                                                                              << 4));
        bf[j][0] = v.x, bf[j][1] = v.y, bf[j][2] = v.z, bf[j][3] = v.w;
        const float4 e = *reinterpret_cast<const float4 *>(stage + L::kOffDc + (((bb * 2 + j) * 4 + t4) << 4));
        da[j] = make_float2(e.x, e.y);
        ss[j] = make_float2(e.z, e.w);
    }
    const uint8_t *rlo = wpiece + g * kRowBytes;  // row g of the tile
    const uint8_t *rhi = rlo + 8 * kRowBytes;      // row g + 8
    const uint2 clo = W::template codes<BB>(rlo, t4), chi = W::template codes<BB>(rhi, t4);
    uint32_t a0[4], a1[4];  // per MMA step: {row g lo, row g+8 lo, row g hi, row g+8 hi}
    q8::i8x4_to_f16x4(clo.x, a0[0], a0[2]);
    q8::i8x4_to_f16x4(chi.x, a0[1], a0[3]);
    q8::i8x4_to_f16x4(clo.y, a1[0], a1[2]);
    q8::i8x4_to_f16x4(chi.y, a1[1], a1[3]);
    const float dlo = W::template d<BB>(rlo), dhi = W::template d<BB>(rhi);
    const float mlo = W::template m<BB>(rlo), mhi = W::template m<BB>(rhi);
    // the token tiles' first k-halves, then their second halves: consecutive
    // MMAs are independent when NT > 1
    float c[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        c[j][0] = c[j][1] = c[j][2] = c[j][3] = 0.0f;
        mma_f16_16816(c[j], a0, bf[j][0], bf[j][1]);
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) mma_f16_16816(c[j], a1, bf[j][2], bf[j][3]);
#pragma unroll
    for (int j = 0; j < NT; ++j) sb_epilogue<W>(acc[j], c[j], dlo, dhi, mlo, mhi, da[j], ss[j]);
}

__device__ __forceinline__ void mma_s8_16832(int (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same block for one token tile (t <= 8) on the int8 MMA: the codes enter
// the tensor core as they are, with no widening, and the s32 result is the
// same exact block dot.  One m16n8k32 covers the block: code words t4 and
// t4 + 4 are its k ranges 4*t4.. and 16 + 4*t4.. for A and B alike.  One
// tile needs about half of the int8 MMA rate at HBM speed; two tiles would
// need more than all of it, so t > 8 keeps the f16 step.
template <class W, int BB, int NT>
__device__ __forceinline__ void sb_block_s8(const uint8_t *wpiece, const uint8_t *stage, int pc, int g, int t4,
                                            const float2 (&da)[NT], const float2 (&ss)[NT], float2 (&acc)[NT][2])
{
    constexpr int kRowBytes = SbLayout<W>::kRowBytes;
    const uint8_t *rlo = wpiece + g * kRowBytes;  // row g of the tile
    const uint8_t *rhi = rlo + 8 * kRowBytes;      // row g + 8
    const uint2 clo = W::template codes<BB>(rlo, t4), chi = W::template codes<BB>(rhi, t4);
    const float dlo = W::template d<BB>(rlo), dhi = W::template d<BB>(rhi);
    const float mlo = W::template m<BB>(rlo), mhi = W::template m<BB>(rhi);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const uint2 v = sb_act<BB>(stage, pc, 8 * j + g, t4);
        int ci[4] = {0, 0, 0, 0};
        mma_s8_16832(ci, clo.x, chi.x, clo.y, chi.y, v.x, v.y);
        const float c[4] = {static_cast<float>(ci[0]), static_cast<float>(ci[1]), static_cast<float>(ci[2]),
                            static_cast<float>(ci[3])};
        sb_epilogue<W>(acc[j], c, dlo, dhi, mlo, mhi, da[j], ss[j]);
    }
}

// d_a of block BB from a token's eight d|ssum words of the stage
__device__ __forceinline__ float sb_half_lo(uint32_t w)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu)));
}

template <class W, int BB, int NT>
__device__ __forceinline__ void sb_step(const uint8_t *wpiece, const uint8_t *stage, int pc, int g, int t4,
                                        const uint4 (&dsv)[NT][2][2], float2 (&acc)[NT][2])
{
    if constexpr (NT > Q8_SB_S8_TILES) {
        sb_block<W, BB, NT>(wpiece, stage, pc, g, t4, acc);  // the prepared f16 activation
    } else {
        float2 da[NT], ss[NT];  // d_a and (asymmetric weights) the plane's ssum of the token pair
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            const uint4 &e = dsv[j][0][BB >> 2], &o = dsv[j][1][BB >> 2];  // tokens 8j + 2*t4, 8j + 2*t4 + 1
            constexpr int q = BB & 3;
            const uint32_t we = q == 0 ? e.x : q == 1 ? e.y : q == 2 ? e.z : e.w;
            const uint32_t wo = q == 0 ? o.x : q == 1 ? o.y : q == 2 ? o.z : o.w;
            da[j] = make_float2(sb_half_lo(we), sb_half_lo(wo));
            ss[j] = make_float2(static_cast<float>(static_cast<int16_t>(we >> 16)),
                                static_cast<float>(static_cast<int16_t>(wo >> 16)));
        }
        sb_block_s8<W, BB, NT>(wpiece, stage, pc, g, t4, da, ss, acc);
    }
}

// The f16 path's activation, prepared once per stage by the consumer warps
// together (thread u of kSbWarps * 32) instead of by each warp per block: per
// item (block, token, t4) the code words t4 and t4 + 4 of the token's block
// (TMA box 2*pc + BB/4, 128-byte swizzled) widened exactly to four f16 pairs
// at item * 16 of the f16 area; per item (block, token tile j, t4) the d_a
// and ssum of tokens 8j + 2*t4 and 8j + 2*t4 + 1.
template <class W>
__device__ __forceinline__ void sb_prep_act(uint8_t *stage, int u)
{
    using L = SbLayout<W>;
    constexpr int kItems = kSbPieces * kSbGroup * kSbMaxTokens * 4;
#pragma unroll
    for (int it = u; it < kItems; it += kSbWarps * 32) {
        const int t4 = it & 3, tok = (it >> 2) & (kSbMaxTokens - 1), bb = it >> 6;
        const int pc = bb / kSbGroup, BB = bb % kSbGroup;
        const int c0 = 2 * (BB & 3);
        const uint8_t *line = stage + kSbOffAct + (2 * pc + (BB >> 2)) * 2048 + tok * 128;
        const uint32_t lo = *reinterpret_cast<const uint32_t *>(line + ((c0 ^ (tok & 7)) << 4) + 4 * t4);
        const uint32_t hi = *reinterpret_cast<const uint32_t *>(line + (((c0 + 1) ^ (tok & 7)) << 4) + 4 * t4);
        uint4 v;
        q8::i8x4_to_f16x4(lo, v.x, v.y);
        q8::i8x4_to_f16x4(hi, v.z, v.w);
        *reinterpret_cast<uint4 *>(stage + L::kOffAh + (it << 4)) = v;
    }
    constexpr int kScaleItems = kSbPieces * kSbGroup * 2 * 4;
    static_assert(kScaleItems <= kSbWarps * 32, "one scale item per thread at most");
    if (u < kScaleItems) {
        const int t4 = u & 3, j = (u >> 2) & 1, bb = u >> 3;
        const int pc = bb / kSbGroup, BB = bb % kSbGroup;
        const uint8_t *dw = stage + kSbOffDs + 4 * kSbGroup * pc + 4 * BB;
        const uint32_t w0 = *reinterpret_cast<const uint32_t *>(dw + (8 * j + 2 * t4) * (32 * kSbPieces));
        const uint32_t w1 = *reinterpret_cast<const uint32_t *>(dw + (8 * j + 2 * t4 + 1) * (32 * kSbPieces));
        *reinterpret_cast<float4 *>(stage + L::kOffDc + (u << 4)) =
            make_float4(sb_half_lo(w0), sb_half_lo(w1), static_cast<float>(static_cast<int16_t>(w0 >> 16)),
                        static_cast<float>(static_cast<int16_t>(w1 >> 16)));
    }
}

// Named barrier `id` of `n` threads that also reports whether p held on every
// one of them (all participants get the same answer).
__device__ __forceinline__ bool bar_all(int id, int n, bool p)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.and.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(p)), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// The projections of one small-batch launch (they share the activation and k):
// per projection its weight map, row count, output and first row tile in the
// launch's tile order; tile_begin[count] is the total.
struct SbGroup {
    CUtensorMap w[kMaxProj];
    float *y[kMaxProj];
    int64_t n[kMaxProj];
    int tile_begin[kMaxProj + 1];
    int count;
};

template <class W, int NT>
__global__ void __launch_bounds__(kSbThreads, 2)
gemv_small_kernel(const __grid_constant__ SbGroup grp, const __grid_constant__ CUtensorMap tmQ,
                  const __grid_constant__ CUtensorMap tmD, int nb, int t)
{
    using L = SbLayout<W>;
    constexpr int kSbOffBar = L::kOffBar, kSbStageBytes = L::kStageBytes, kSbStageTx = L::kStageTx;
    constexpr int kSbRowBytes = L::kRowBytes, kSbPieceBytes = L::kPieceBytes;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_base = q8::smem_u32(smem_raw);
    uint8_t *ring = smem_raw + (((raw_base + 1023u) & ~1023u) - raw_base);  // 1024-byte aligned (swizzle atoms)
    cg::cluster_group cluster = cg::this_cluster();
    const int ks = static_cast<int>(cluster.num_blocks());  // CTAs splitting k (the cluster spans x only)
    const int rank = static_cast<int>(cluster.block_rank());
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + kSbOffBar);  // [stage]: the stage's boxes landed
    uint64_t *empty = full + kSbStages;                                 // [stage]: consumer warps done
    volatile int *bad = reinterpret_cast<volatile int *>(ring + kSbOffBar + kSbStages * 16);
    // this CTA's projection and first row (found where needed, not held across the main loop)
    auto locate = [&](int &pi) -> int64_t {
        const int rtile = static_cast<int>(blockIdx.x) / ks;  // row tile of the launch, over all projections
        pi = 0;
#pragma unroll
        for (int i = 1; i < kMaxProj; ++i)
            if (i < grp.count && rtile >= grp.tile_begin[i]) pi = i;
        return static_cast<int64_t>(rtile - grp.tile_begin[pi]) * kSbRows;
    };
    // the last stage may hang past the end of the rows: those pieces, codes
    // and scales arrive as zeros and add exactly nothing
    const int stages_total = (nb + kSbGroup * kSbPieces - 1) / (kSbGroup * kSbPieces);
    const int gc0 = static_cast<int>(static_cast<int64_t>(stages_total) * rank / ks);  // this CTA's share of k
    const int ng = static_cast<int>(static_cast<int64_t>(stages_total) * (rank + 1) / ks) - gc0;

    q8::griddep_launch_dependents();
    if (threadIdx.x == 0) {
        *bad = 0;
        for (int s = 0; s < kSbStages; ++s) {
            q8::mbar_init(&full[s], 1);
            q8::mbar_init(&empty[s], kSbWarps);
        }
        q8::fence_mbar_init();
    }
    __syncthreads();

    if (warp == kSbWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            // The weights do not depend on the previous kernel in the stream:
            // the first stages' weight boxes go out before waiting for it
            // (programmatic dependent launch), every activation box after.
            const uint32_t rb = q8::smem_u32(ring);
            int pi;
            const int64_t row0 = locate(pi);
            const CUtensorMap *tmW = &grp.w[pi];
            auto issue_w = [&](int s, int gi) {
                q8::mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(kSbStageTx));
                q8::tma_load_3d(rb + s * kSbStageBytes + kSbOffW, tmW, 0, gi * kSbPieces, static_cast<int>(row0),
                                q8::smem_u32(&full[s]));
            };
            auto issue_a = [&](int s, int gi) {
                const uint32_t st = rb + s * kSbStageBytes;
#pragma unroll
                for (int b = 0; b < 2 * kSbPieces; ++b)
                    q8::tma_load_2d(st + kSbOffAct + 2048 * b, &tmQ, gi * (256 * kSbPieces) + 128 * b, 0,
                                    q8::smem_u32(&full[s]));
                q8::tma_load_2d(st + kSbOffDs, &tmD, gi * (kSbGroup * kSbPieces), 0, q8::smem_u32(&full[s]));
            };
            int i = 0;
            for (; i < kSbStages && i < ng; ++i) issue_w(i, gc0 + i);
            q8::griddep_wait();
            for (int s = 0; s < i; ++s) issue_a(s, gc0 + s);
            for (; i < ng; ++i) {
                const int s = i % kSbStages;
                if (!q8::mbar_wait_bounded(&empty[s], static_cast<uint32_t>(i / kSbStages - 1) & 1u)) {
                    atomicOr(&g_gemv_err, 1u);
                    *bad = 1;
                    break;
                }
                issue_w(s, gc0 + i);
                issue_a(s, gc0 + i);
            }
            // let every issued stage land (bounded) before the CTA can exit
            for (int j = (i > kSbStages ? i - kSbStages : 0); j < i; ++j)
                if (!q8::mbar_wait_bounded(&full[j % kSbStages], static_cast<uint32_t>(j / kSbStages) & 1u,
                                           Q8_DRAIN_LIMIT_NS)) {
                    atomicOr(&g_gemv_err, 1u);
                    *bad = 1;
                }
        }
    }
    float2 acc[NT][2];  // [token tile][row g, row g+8]: tokens 2*t4, 2*t4+1
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = make_float2(0.0f, 0.0f);
    const int tile = warp % kSbTiles, pc = warp / kSbTiles;  // this warp's 16 rows and piece
    if (warp < kSbWarps) {
        // ------------------------------------------------------------ consumers
        const int g = lane >> 2, t4 = lane & 3;
        for (int i = 0; i < ng; ++i) {
            const int s = i % kSbStages;
            const bool got = q8::mbar_wait_bounded(&full[s], static_cast<uint32_t>(i / kSbStages) & 1u);
            uint8_t *st = ring + s * kSbStageBytes;
            uint4 dsv[NT][2][2];  // [tile][token 2*t4 + e][blocks 0-3, 4-7]: the stage's d|ssum words (int8 path)
            if constexpr (NT > Q8_SB_S8_TILES) {
                // f16 path: the consumer warps prepare the stage's activation together;
                // the barrier publishes it and tells every warp whether all stages arrived
                if (got) sb_prep_act<W>(st, static_cast<int>(threadIdx.x));
                __syncwarp();  // the barrier below is warp-aligned; got may differ between lanes on a timeout
                if (!bar_all(1, kSbWarps * 32, got)) {
                    if (lane == 0) {
                        atomicOr(&g_gemv_err, 1u);
                        *bad = 1;
                    }
                    break;
                }
            } else {
                if (!__all_sync(Q8_FULL_MASK, got)) {
                    if (lane == 0) {
                        atomicOr(&g_gemv_err, 1u);
                        *bad = 1;
                    }
                    break;
                }
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const uint4 *dw = reinterpret_cast<const uint4 *>(st + kSbOffDs + 4 * kSbGroup * pc +
                                                                          (8 * j + 2 * t4 + e) * (32 * kSbPieces));
                        dsv[j][e][0] = dw[0];
                        dsv[j][e][1] = dw[1];
                    }
            }
            const uint8_t *wp = st + kSbOffW + tile * 16 * kSbRowBytes + pc * kSbPieceBytes;
            sb_step<W, 0, NT>(wp, st, pc, g, t4, dsv, acc);
            sb_step<W, 1, NT>(wp, st, pc, g, t4, dsv, acc);
            sb_step<W, 2, NT>(wp, st, pc, g, t4, dsv, acc);
            sb_step<W, 3, NT>(wp, st, pc, g, t4, dsv, acc);
            sb_step<W, 4, NT>(wp, st, pc, g, t4, dsv, acc);
            sb_step<W, 5, NT>(wp, st, pc, g, t4, dsv, acc);
            sb_step<W, 6, NT>(wp, st, pc, g, t4, dsv, acc);
            sb_step<W, 7, NT>(wp, st, pc, g, t4, dsv, acc);
            __syncwarp();
            if (lane == 0) q8::mbar_arrive(&empty[s]);
        }
    }
    __syncthreads();  // the ring is consumed and every box has landed: reuse it for the partial sums
    float *part = reinterpret_cast<float *>(ring);  // [piece][token 16][row]
    if (warp < kSbWarps) {
        const int g = lane >> 2, t4 = lane & 3;
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int r = tile * 16 + g + 8 * e;
                part[(pc * kSbMaxTokens + 8 * j + 2 * t4) * kSbRows + r] = acc[j][e].x;
                part[(pc * kSbMaxTokens + 8 * j + 2 * t4 + 1) * kSbRows + r] = acc[j][e].y;
            }
    }
    __syncthreads();
    // this CTA's sum over its pieces, in piece order, into piece 0's slot
    for (int o = threadIdx.x; o < 8 * NT * kSbRows; o += kSbThreads) {
        float v = part[o];
#pragma unroll
        for (int p = 1; p < kSbPieces; ++p) v += part[p * kSbMaxTokens * kSbRows + o];
        part[o] = v;
    }
    cluster.sync();  // every CTA's partial sums are in its shared memory
    // Each CTA of the cluster finishes a 1/ks share of the tile's outputs: it
    // loads the ks partial sums of an output together (distributed shared
    // memory) and adds them in rank order.
    bool any_bad = false;
    for (int r = 0; r < ks; ++r) any_bad |= *cluster.map_shared_rank(const_cast<int *>(bad), r) != 0;
    if (!any_bad) {
        int pi;
        const int64_t row0 = locate(pi);
        const int64_t n = grp.n[pi];
        float *__restrict__ y = grp.y[pi];
        const int rows = static_cast<int>(min(static_cast<int64_t>(kSbRows), n - row0));
        constexpr int kOut = 8 * NT * kSbRows;
        const int share = (kOut + ks - 1) / ks;
        const int o_end = min(kOut, (rank + 1) * share);
        const float *src[kSbMaxCluster];
#pragma unroll
        for (int pr = 0; pr < kSbMaxCluster; ++pr) src[pr] = pr < ks ? cluster.map_shared_rank(part, pr) : part;
        for (int o = rank * share + static_cast<int>(threadIdx.x); o < o_end; o += kSbThreads) {
            const int tok = o / kSbRows, r = o % kSbRows;
            if (tok < t && r < rows) {
                float pv[kSbMaxCluster];
#pragma unroll
                for (int pr = 0; pr < kSbMaxCluster; ++pr) pv[pr] = pr < ks ? src[pr][o] : 0.0f;
                float v = pv[0];
#pragma unroll
                for (int pr = 1; pr < kSbMaxCluster; ++pr)
                    if (pr < ks) v += pv[pr];
                y[tok * n + row0 + r] = v;
            }
        }
    }
    cluster.sync();  // every CTA keeps its shared memory until its peers have read it
}

int ceil_log2(int v)
{
    int l = 0;
    while ((1 << l) < v) ++l;
    return l;
}

} // namespace

namespace q8 {

int gemv_take_error(cudaStream_t s)
{
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbolAsync(&v, g_gemv_err, sizeof(v), 0, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyToSymbolAsync(g_gemv_err, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return Q8_ERR_CUDA;
    return v ? Q8_ERR_DEVICE_TIMEOUT : Q8_OK;
}

// Launch the generic kernel for `tokens` plane rows (used by the GEMM too).
int gemv_generic_launch(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, float *y,
                        int64_t tokens, cudaStream_t s)
{
    const int nb = static_cast<int>(k / 32);
    const int lpr_log2 = min(5, ceil_log2(nb));
    const int rpw = 32 >> lpr_log2;
    const int64_t warps = (n + rpw - 1) / rpw;
    const dim3 grid(static_cast<unsigned>((warps + 3) / 4), static_cast<unsigned>(tokens));
    return launch_pdl(gemv_generic_kernel, grid, dim3(128), 0, s, static_cast<const uint8_t *>(w), n, nb, qs, ds, y,
                      lpr_log2);
}

} // namespace q8

namespace {

// Launch the small-batch kernel for weight format W over `count` projections
// of one activation: 1 <= tokens <= 16, (k/32) % 8 == 0.  Their row tiles form
// one grid (small projections ride along with large ones).  The cluster size
// (CTAs splitting k, 1..8) makes the grid about one wave of the CTAs that fit
// on the GPU at once (the occupancy the runtime reports for this kernel, its
// shared memory and its registers).
template <class W>
int gemv_small_launch_t(const q8_gemv_proj *projs, int count, int64_t k, const int8_t *qs, const uint32_t *ds,
                        int64_t tokens, cudaStream_t s, int slot1, int slot2)
{
    using L = SbLayout<W>;
    const int64_t nb = k / 32;
    if (count < 1 || count > kMaxProj || tokens < 1 || tokens > kSbMaxTokens || nb % kSbGroup != 0 ||
        nb > (int64_t(1) << 30))
        return Q8_ERR_ARG;
    const int64_t stages = (nb + kSbGroup * kSbPieces - 1) / (kSbGroup * kSbPieces);
    const int sms = q8::device_sm_count();
    if (sms <= 0) return Q8_ERR_DEVICE;
    const bool wide = tokens > 8;
    const void *fn = wide ? reinterpret_cast<const void *>(gemv_small_kernel<W, 2>)
                          : reinterpret_cast<const void *>(gemv_small_kernel<W, 1>);
    if (!q8::set_max_dynamic_smem(fn, L::kSmem, wide ? slot2 : slot1)) return Q8_ERR_LAUNCH;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kSbThreads, static_cast<size_t>(L::kSmem)) !=
            cudaSuccess ||
        per_sm < 1)
        return Q8_ERR_LAUNCH;
    SbGroup grp;
    std::memset(&grp, 0, sizeof(grp));
    grp.count = count;
    int64_t tiles = 0;
    for (int i = 0; i < count; ++i) {
        grp.tile_begin[i] = static_cast<int>(tiles);
        tiles += (projs[i].n + kSbRows - 1) / kSbRows;
        if (tiles > 0x7fffffff) return Q8_ERR_ARG;
        grp.y[i] = projs[i].y;
        grp.n[i] = projs[i].n;
        // weights as [n rows][nb/8 pieces][piece bytes / 2 u16]; box = kSbRows rows x kSbPieces pieces
        if (!q8::make_map_3d(&grp.w[i], CU_TENSOR_MAP_DATA_TYPE_UINT16, projs[i].w, L::kPieceBytes / 2,
                             static_cast<uint64_t>(nb / kSbGroup), static_cast<uint64_t>(projs[i].n), L::kPieceBytes,
                             static_cast<uint64_t>(nb * W::kBlockBytes), L::kPieceBytes / 2, kSbPieces, kSbRows,
                             CU_TENSOR_MAP_SWIZZLE_NONE))
            return Q8_ERR_LAUNCH;
    }
    for (int i = count; i <= kMaxProj; ++i) grp.tile_begin[i] = static_cast<int>(tiles);
    // about one wave of resident CTAs, at least one stage per CTA
    int64_t ks = (static_cast<int64_t>(per_sm) * sms) / tiles;
    ks = ks < 1 ? 1 : (ks > kSbMaxCluster ? kSbMaxCluster : ks);
    if (ks > stages) ks = stages;
    if (tiles * ks > 0x7fffffff) return Q8_ERR_ARG;
    const dim3 grid(static_cast<unsigned>(tiles * ks));
    CUtensorMap mq, md;
    if (!q8::make_map_2d(&mq, CU_TENSOR_MAP_DATA_TYPE_UINT8, qs, static_cast<uint64_t>(k), static_cast<uint64_t>(tokens),
                         static_cast<uint64_t>(k), 128, kSbMaxTokens, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !q8::make_map_2d(&md, CU_TENSOR_MAP_DATA_TYPE_UINT32, ds, static_cast<uint64_t>(nb), static_cast<uint64_t>(tokens),
                         static_cast<uint64_t>(nb * 4), kSbGroup * kSbPieces, kSbMaxTokens, CU_TENSOR_MAP_SWIZZLE_NONE))
        return Q8_ERR_LAUNCH;
    if (wide)
        return q8::launch_pdl_cluster(gemv_small_kernel<W, 2>, grid, dim3(kSbThreads), L::kSmem, s, static_cast<int>(ks),
                                      grp, mq, md, static_cast<int>(nb), static_cast<int>(tokens));
    return q8::launch_pdl_cluster(gemv_small_kernel<W, 1>, grid, dim3(kSbThreads), L::kSmem, s, static_cast<int>(ks),
                                  grp, mq, md, static_cast<int>(nb), static_cast<int>(tokens));
}

} // namespace

namespace q8 {

int gemv_small_launch(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, float *y,
                      int64_t tokens, cudaStream_t s)
{
    const q8_gemv_proj p = {w, n, y};
    return gemv_small_launch_t<SbQ8_0>(&p, 1, k, qs, ds, tokens, s, 3, 4);
}

int gemv_small_grouped_launch(const q8_gemv_proj *projs, int count, int64_t k, const int8_t *qs, const uint32_t *ds,
                              int64_t tokens, cudaStream_t s)
{
    return gemv_small_launch_t<SbQ8_0>(projs, count, k, qs, ds, tokens, s, 3, 4);
}

int gemv_small_q4a_launch(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, float *y,
                          int64_t tokens, cudaStream_t s)
{
    const q8_gemv_proj p = {w, n, y};
    return gemv_small_launch_t<SbQ4A>(&p, 1, k, qs, ds, tokens, s, 7, 8);
}

int gemv_small_q4a_grouped_launch(const q8_gemv_proj *projs, int count, int64_t k, const int8_t *qs,
                                  const uint32_t *ds, int64_t tokens, cudaStream_t s)
{
    return gemv_small_launch_t<SbQ4A>(projs, count, k, qs, ds, tokens, s, 7, 8);
}

} // namespace q8

namespace {

// Launch the staged kernel for `count` projections of one activation.
// SwiGLU pairing output of a gate/up launch (plane row 0 of silu(gate) * up).
struct GvPair {
    int8_t *qs;
    uint32_t *ds;
};

template <class F>
int gemv_staged_launch(const q8_gemv_proj *projs, int count, int64_t k, const int8_t *qs, const uint32_t *ds,
                       cudaStream_t s, int smem_slot, const GvAct *act = nullptr, const GvPair *pair = nullptr)
{
    constexpr int kStages = F::kStages;
    constexpr int kMaxWarps = F::kWarps;
    constexpr int kPieceBytes = 32 * F::kLaneChunks * F::kChunkBytes;
    constexpr int kPieceChunks = 32 * F::kLaneChunks;
    const int64_t nb = k / 32;
    GvGeom g;
    if (act) {
        g.act = *act;
    } else {
        g.act = GvAct{};  // producer 0: stage plane row 0
    }
    g.count = count;
    g.nc = static_cast<int>(nb / 4);
    if (g.nc > 32) {  // long rows: one row per piece, 32*J chunks of it
        g.lpr_log2 = 5;
        g.rpw = 1;
        g.ppr = (g.nc + kPieceChunks - 1) / kPieceChunks;
    } else {          // short rows: J slots of 32 >> lpr_log2 whole rows
        g.lpr_log2 = ceil_log2(g.nc);
        g.rpw = F::kLaneChunks * (32 >> g.lpr_log2);
        g.ppr = 1;
    }
    int64_t groups = 0;
    for (int i = 0; i < kMaxProj; ++i) {
        if (i < count) {
            g.p[i].w = static_cast<const uint8_t *>(projs[i].w);
            g.p[i].y = projs[i].y;
            g.p[i].n = projs[i].n;
            g.p[i].g_begin = groups;
            groups += (projs[i].n + g.rpw - 1) / g.rpw;
        } else {
            g.p[i].w = nullptr;
            g.p[i].y = nullptr;
            g.p[i].n = 0;
            g.p[i].g_begin = groups;
        }
    }
    g.groups = groups;
    g.pair_upc = 0;
    g.pair_qs = pair ? pair->qs : nullptr;
    g.pair_ds = pair ? pair->ds : nullptr;
    if (pair && (count != 2 || g.rpw != 1 || projs[0].n != projs[1].n || projs[0].n % 32 != 0)) return Q8_ERR_ARG;
    const int sms = q8::device_sm_count();
    if (sms <= 0) return Q8_ERR_DEVICE;
    // warps per CTA: enough to spread the row groups over every SM, at most
    // kMaxWarps, and no more rings than fit beside the staged activation
    constexpr int kSmemCap = 227 * 1024;
    const int act_bytes = (g.nc * kActChunkBytes + 127) & ~127;
    const int64_t fit = (kSmemCap - smem_header_bytes<F>() - act_bytes) / (kStages * kPieceBytes);
    static_assert(kSmemCap - kMaxWarps * kStages * 16 - 128 - kMaxActChunks * kActChunkBytes >= 4 * kStages * kPieceBytes,
                  "at least four warps' rings fit beside the longest staged activation");
    static_assert(kMaxWarps * 32 <= 1024, "threads per CTA");
    int64_t nw = (g.groups + sms - 1) / sms;
    nw = nw < 1 ? 1 : (nw > kMaxWarps ? kMaxWarps : nw);
    nw = nw > fit ? fit : nw;
    int64_t grid = (g.groups + nw - 1) / nw;
    grid = grid > sms ? sms : grid;
    if (pair) {  // whole 64-row units per CTA, and their buffer beside the activation
        const int64_t units = g.groups / 64;
        int64_t upc = (units + grid - 1) / grid;
        const int64_t fit2 = (kSmemCap - smem_header_bytes<F>() - act_bytes -
                              pair_region_bytes(static_cast<int>(upc))) / (kStages * kPieceBytes);
        if (upc > 4096 || fit2 < 1) return Q8_ERR_ARG;
        if (nw > fit2) {  // fewer warps: more CTAs, so no more units per CTA than reserved
            nw = fit2;
            grid = (g.groups + nw - 1) / nw;
            grid = grid > sms ? sms : grid;
            upc = (units + grid - 1) / grid;
        }
        g.pair_upc = static_cast<int>(upc);
    }
    const int smem = smem_header_bytes<F>() + act_bytes + pair_region_bytes(g.pair_upc) +
                     static_cast<int>(nw) * kStages * kPieceBytes;
    if (!q8::set_max_dynamic_smem(reinterpret_cast<const void *>(gemv_staged_kernel<F>), kSmemCap, smem_slot))
        return Q8_ERR_LAUNCH;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(static_cast<unsigned>(nw * 32));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // may start before the producer ends
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, gemv_staged_kernel<F>, reinterpret_cast<const uint4 *>(qs), ds, g) != cudaSuccess)
        return Q8_ERR_LAUNCH;
    return q8::launch_status();
}

int check_projs(const q8_gemv_proj *projs, int count, int64_t k)
{
    if (!projs || count < 1 || count > Q8_MAX_GROUP || k <= 0 || (k % 32) != 0) return Q8_ERR_ARG;
    for (int i = 0; i < count; ++i)
        if (!projs[i].w || !projs[i].y || projs[i].n < 1 || projs[i].n > (int64_t(1) << 40)) return Q8_ERR_ARG;
    for (int i = 0; i < count; ++i)
        if (!q8::aligned16(projs[i].w) || !q8::aligned16(projs[i].y)) return Q8_ERR_ALIGN;
    return Q8_OK;
}

int check_gemv_args(const q8_gemv_proj *projs, int count, int64_t k, const int8_t *qs, const uint32_t *ds)
{
    if (!qs || !ds) return Q8_ERR_ARG;
    const int st = check_projs(projs, count, k);
    if (st != Q8_OK) return st;
    if (!q8::aligned16(qs) || !q8::aligned16(ds)) return Q8_ERR_ALIGN;
    return Q8_OK;
}

int gemv_dispatch(const q8_gemv_proj *projs, int count, int64_t k, const int8_t *qs, const uint32_t *ds, void *stream)
{
    int st = check_gemv_args(projs, count, k, qs, ds);
    if (st != Q8_OK) return st;
    if (!q8::device_is_sm103()) return Q8_ERR_DEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int64_t nb = k / 32;
    if (nb % 8 != 0 || nb / 4 > kMaxActChunks) {  // generic kernel, one launch per projection
        for (int i = 0; i < count; ++i) {
            st = q8::gemv_generic_launch(projs[i].w, projs[i].n, k, qs, ds, projs[i].y, 1, s);
            if (st != Q8_OK) return st;
        }
        return Q8_OK;
    }
    return gemv_staged_launch<FmtQ8_0>(projs, count, k, qs, ds, s, 0);
}

} // namespace

namespace q8 {

int gemv_staged_q4a_launch(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, float *y,
                           cudaStream_t s)
{
    const q8_gemv_proj p = {w, n, y};
    return gemv_staged_launch<FmtQ4A>(&p, 1, k, qs, ds, s, 6);
}

} // namespace q8

extern "C" int q8_0_gemv(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, float *y,
                         void *stream)
{
    const q8_gemv_proj p = {w, n, y};
    return gemv_dispatch(&p, 1, k, qs, ds, stream);
}

extern "C" int q8_0_gemv_grouped(const q8_gemv_proj *projs, int count, int64_t k, const int8_t *qs,
                                 const uint32_t *ds, void *stream)
{
    return gemv_dispatch(projs, count, k, qs, ds, stream);
}

extern "C" int q8_0_gemv_fused(const q8_gemv_proj *projs, int count, int64_t k, int producer, const float *a,
                               const float *b, const float *norm_w, float eps, void *stream)
{
    if (producer != Q8_PRODUCER_QUANT && producer != Q8_PRODUCER_RMSNORM && producer != Q8_PRODUCER_SWIGLU)
        return Q8_ERR_ARG;
    int st = check_projs(projs, count, k);
    if (st != Q8_OK) return st;
    if (!a || (producer == Q8_PRODUCER_SWIGLU && !b) || (producer == Q8_PRODUCER_RMSNORM && !norm_w))
        return Q8_ERR_ARG;
    // the staged path only: whole 8-block row pieces, the row's encoding in
    // shared memory, and (RMSNorm) the standalone kernel's row limit
    if ((k / 32) % 8 != 0 || k / 128 > kMaxActChunks || (producer == Q8_PRODUCER_RMSNORM && k > 32768))
        return Q8_ERR_ARG;
    if (!q8::aligned16(a) || (producer == Q8_PRODUCER_SWIGLU && !q8::aligned16(b)) ||
        (producer == Q8_PRODUCER_RMSNORM && !q8::aligned16(norm_w)))
        return Q8_ERR_ALIGN;
    if (!q8::device_is_sm103()) return Q8_ERR_DEVICE;
    GvAct act{};
    act.producer = producer;
    act.a = reinterpret_cast<const float4 *>(a);
    act.b = producer == Q8_PRODUCER_SWIGLU ? reinterpret_cast<const float4 *>(b) : nullptr;
    act.w = producer == Q8_PRODUCER_RMSNORM ? reinterpret_cast<const float4 *>(norm_w) : nullptr;
    act.eps = eps;
    // one row: the standalone RMSNorm's mapping for rows_pad <= the SM count
    q8::rms_row_mapping(static_cast<int>(k / 4), q8::kRmsMaxThreadsOneRow, act.rms_j, act.rms_p);
    return gemv_staged_launch<FmtQ8_0>(projs, count, k, nullptr, nullptr, static_cast<cudaStream_t>(stream), 0,
                                       &act);
}

extern "C" int q8_0_gemv_gate_up(const void *w_gate, const void *w_up, int64_t nf, int64_t k, const int8_t *qs,
                                 const uint32_t *ds, int producer, const float *a, const float *norm_w, float eps,
                                 float *y_gate, float *y_up, int8_t *qs_out, uint32_t *ds_out, void *stream)
{
    if (!w_gate || !w_up || !qs_out || !ds_out || nf < 32 || nf % 32 != 0 || nf > (int64_t(1) << 40) || k <= 0 ||
        (k % 32) != 0)
        return Q8_ERR_ARG;
    if (producer == 0 ? (!qs || !ds)
                      : ((producer != Q8_PRODUCER_QUANT && producer != Q8_PRODUCER_RMSNORM) || !a ||
                         (producer == Q8_PRODUCER_RMSNORM && (!norm_w || k > 32768))))
        return Q8_ERR_ARG;
    // the staged path with whole rows per warp (more than 16 chunks of 4 blocks)
    if ((k / 32) % 8 != 0 || k / 128 > kMaxActChunks || k / 128 <= 16) return Q8_ERR_ARG;
    if (!q8::aligned16(w_gate) || !q8::aligned16(w_up) || !q8::aligned16(qs_out) || !q8::aligned16(ds_out) ||
        (y_gate && !q8::aligned16(y_gate)) || (y_up && !q8::aligned16(y_up)))
        return Q8_ERR_ALIGN;
    if (producer == 0 ? (!q8::aligned16(qs) || !q8::aligned16(ds))
                      : (!q8::aligned16(a) || (producer == Q8_PRODUCER_RMSNORM && !q8::aligned16(norm_w))))
        return Q8_ERR_ALIGN;
    if (!q8::device_is_sm103()) return Q8_ERR_DEVICE;
    const q8_gemv_proj projs[2] = {{w_gate, nf, y_gate}, {w_up, nf, y_up}};
    const GvPair pair{qs_out, ds_out};
    GvAct act{};
    if (producer != 0) {
        act.producer = producer;
        act.a = reinterpret_cast<const float4 *>(a);
        act.w = producer == Q8_PRODUCER_RMSNORM ? reinterpret_cast<const float4 *>(norm_w) : nullptr;
        act.eps = eps;
        q8::rms_row_mapping(static_cast<int>(k / 4), q8::kRmsMaxThreadsOneRow, act.rms_j, act.rms_p);
    }
    return gemv_staged_launch<FmtQ8_0>(projs, 2, k, producer == 0 ? qs : nullptr, producer == 0 ? ds : nullptr,
                                       static_cast<cudaStream_t>(stream), 0, &act, &pair);
}

extern "C" int q8_0_gemv_batched(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds,
                                 int64_t tokens, float *y, void *stream)
{
    if (!w || !qs || !ds || !y || n < 1 || n > (int64_t(1) << 40) || k <= 0 || (k % 32) != 0 || tokens < 1 ||
        tokens > Q8_GEMV_MAX_TOKENS)
        return Q8_ERR_ARG;
    if (!q8::aligned16(w) || !q8::aligned16(qs) || !q8::aligned16(ds) || !q8::aligned16(y)) return Q8_ERR_ALIGN;
    if (!q8::device_is_sm103()) return Q8_ERR_DEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((k / 32) % 8 != 0) return q8::gemv_generic_launch(w, n, k, qs, ds, y, tokens, s);
    return q8::gemv_small_launch(w, n, k, qs, ds, y, tokens, s);
}

extern "C" int q8_0_gemv_batched_grouped(const q8_gemv_proj *projs, int count, int64_t k, const int8_t *qs,
                                         const uint32_t *ds, int64_t tokens, void *stream)
{
    if (!projs || count < 1 || count > kMaxProj || !qs || !ds || k <= 0 || (k % 32) != 0 || tokens < 1 ||
        tokens > Q8_GEMV_MAX_TOKENS)
        return Q8_ERR_ARG;
    for (int i = 0; i < count; ++i)
        if (!projs[i].w || !projs[i].y || projs[i].n < 1 || projs[i].n > (int64_t(1) << 40)) return Q8_ERR_ARG;
    if (!q8::aligned16(qs) || !q8::aligned16(ds)) return Q8_ERR_ALIGN;
    for (int i = 0; i < count; ++i)
        if (!q8::aligned16(projs[i].w) || !q8::aligned16(projs[i].y)) return Q8_ERR_ALIGN;
    if (!q8::device_is_sm103()) return Q8_ERR_DEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((k / 32) % 8 == 0) return q8::gemv_small_grouped_launch(projs, count, k, qs, ds, tokens, s);
    for (int i = 0; i < count; ++i) {
        const int st = q8::gemv_generic_launch(projs[i].w, projs[i].n, k, qs, ds, projs[i].y, tokens, s);
        if (st != Q8_OK) return st;
    }
    return Q8_OK;
}
