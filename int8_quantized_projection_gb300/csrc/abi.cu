// abi.cu -- C ABI plumbing of libq8proj: device checks, status codes,
// q8_check, and the GEMM dispatch by shape.
#include <mutex>

#include "q8_common.cuh"

namespace q8 {

namespace {
constexpr int kMaxDevices = 64;
constexpr int kMaxSlots = 20;
int g_sms[kMaxDevices];        // 0 = not queried yet
int g_is103[kMaxDevices];      // 0 = unknown, 1 = yes, 2 = no
int g_smem_set[kMaxDevices][kMaxSlots];
std::mutex g_mu;

int current_device()
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

void query(int dev)
{
    cudaDeviceProp p;
    if (cudaGetDeviceProperties(&p, dev) != cudaSuccess) {
        g_sms[dev] = 0;
        g_is103[dev] = 2;
        return;
    }
    g_sms[dev] = p.multiProcessorCount;
    g_is103[dev] = (p.major == 10 && p.minor == 3) ? 1 : 2;
}
} // namespace

int device_sm_count()
{
    const int dev = current_device();
    if (dev < 0) return 0;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_is103[dev] == 0) query(dev);
    return g_sms[dev];
}

bool device_is_sm103()
{
    const int dev = current_device();
    if (dev < 0) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_is103[dev] == 0) query(dev);
    return g_is103[dev] == 1;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (the
// library does not link libcuda); looked up once, thread-safely.
EncodeTiledFn encode_fn()
{
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return nullptr;
    }();
    return fn;
}

bool make_map_2d(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, uint64_t d0, uint64_t d1,
                 uint64_t stride_bytes, uint32_t b0, uint32_t b1, CUtensorMapSwizzle sw)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {d0, d1};
    const cuuint64_t strides[1] = {stride_bytes};
    const cuuint32_t box[2] = {b0, b1};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_3d(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, uint64_t d0, uint64_t d1, uint64_t d2,
                 uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t b0, uint32_t b1, uint32_t b2,
                 CUtensorMapSwizzle sw)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {d0, d1, d2};
    const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
    const cuuint32_t box[3] = {b0, b1, b2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, dt, 3, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool set_max_dynamic_smem(const void *func, int bytes, int slot)
{
    const int dev = current_device();
    if (dev < 0 || slot < 0 || slot >= kMaxSlots) return false;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_smem_set[dev][slot] >= bytes) return true;
    if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
    g_smem_set[dev][slot] = bytes;
    return true;
}

int launch_status()
{
    return cudaGetLastError() == cudaSuccess ? Q8_OK : Q8_ERR_LAUNCH;
}

int gemm_mma_launch(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, int64_t t, float *y,
                    cudaStream_t s);

int gemm_tc_launch(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, int64_t t, float *y,
                   void *workspace, cudaStream_t s);
size_t gemm_workspace_bytes(int64_t n, int64_t t, int64_t k);
size_t gemm_prepared_workspace_bytes(int64_t n, int64_t t, int64_t k);
size_t gemm_prepared_weights_bytes(int64_t n, int64_t k);
int gemm_prepare_weights_launch(const void *w, int64_t n, int64_t k, void *wprep, cudaStream_t s);
int gemm_tc_prepared_launch(const void *wprep, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, int64_t t,
                            float *y, void *workspace, cudaStream_t s);

} // namespace q8

extern "C" int64_t q8_plane_rows(int64_t rows)
{
    if (rows <= 0) return 128;
    return (rows + 127) / 128 * 128;
}

extern "C" const char *q8_strerror(int status)
{
    switch (status) {
    case Q8_OK: return "ok";
    case Q8_ERR_ARG: return "invalid argument (null pointer, size, or k % 32 != 0)";
    case Q8_ERR_ALIGN: return "pointer not 16-byte aligned";
    case Q8_ERR_DEVICE: return "current device is not sm_103 (GB300)";
    case Q8_ERR_LAUNCH: return "kernel launch failed";
    case Q8_ERR_DEVICE_TIMEOUT: return "a bounded on-device wait ran out";
    case Q8_ERR_CUDA: return "CUDA runtime error";
    case Q8_ERR_TOO_BIG: return "request exceeds the fixed scratch of the no-allocation entry point";
    default: return "unknown status";
    }
}

extern "C" int q8_num_sms(void) { return q8::device_sm_count(); }

extern "C" int q8_check(void *stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return Q8_ERR_CUDA;
    const int a = q8::gemv_take_error(s);
    const int b = q8::gemm_take_error(s);
    const int c = q8::quant_take_error(s);
    if (a == Q8_ERR_CUDA || b == Q8_ERR_CUDA || c == Q8_ERR_CUDA) return Q8_ERR_CUDA;
    if (a != Q8_OK) return a;
    if (b != Q8_OK) return b;
    return c;
}

namespace q8 {

int gemv_sliced_launch(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, float *y,
                       int64_t tokens, cudaStream_t s)
{
    const int64_t nb = k / 32;
    for (int64_t c = 0; c < tokens; c += Q8_GEMV_MAX_TOKENS) {  // slice starts stay 16-byte aligned
        const int64_t tt = tokens - c < Q8_GEMV_MAX_TOKENS ? tokens - c : Q8_GEMV_MAX_TOKENS;
        const int st = gemv_small_launch(w, n, k, qs + c * k, ds + c * nb, y + c * n, tt, s);
        if (st != Q8_OK) return st;
    }
    return Q8_OK;
}

} // namespace q8

// The tcgen05 GEMM's grid limits: token tiles of 192 along x, weight-row
// tiles of 128 along y (at most 65535), f16 operand rows addressed in 32 bits.
static bool gemm_tc_shape_ok(int64_t n, int64_t t, int64_t k)
{
    return n <= int64_t(65535) * 128 && t <= (int64_t(1) << 31) - 256 && k <= (int64_t(1) << 31) / 2;
}

extern "C" size_t q8_0_gemm_workspace_bytes(int64_t n, int64_t t, int64_t k)
{
    if (n < 1 || t <= q8::kSlicedMaxTokens || k <= 0 || (k % 32) != 0 || (k / 32) % 8 != 0) return 0;
    return q8::gemm_workspace_bytes(n, t, k);
}

extern "C" int q8_0_gemm(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, int64_t t,
                         int64_t rows_pad, float *y, void *workspace, size_t workspace_bytes, void *stream)
{
    if (!w || !qs || !ds || !y || n < 1 || t < 1 || k <= 0 || (k % 32) != 0 || rows_pad < t) return Q8_ERR_ARG;
    const size_t need = q8_0_gemm_workspace_bytes(n, t, k);
    if (need > 0 && (!workspace || workspace_bytes < need)) return Q8_ERR_ARG;
    if (!q8::aligned16(w) || !q8::aligned16(qs) || !q8::aligned16(ds) || !q8::aligned16(y)) return Q8_ERR_ALIGN;
    if (need > 0 && !q8::aligned16(workspace)) return Q8_ERR_ALIGN;
    if (!q8::device_is_sm103()) return Q8_ERR_DEVICE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (t == 1) return q8_0_gemv(w, n, k, qs, ds, y, stream);
    if ((k / 32) % 8 != 0) {
        if (t > 65535) return Q8_ERR_ARG;  // generic kernel: one grid row per token
        return q8::gemv_generic_launch(w, n, k, qs, ds, y, t, s);
    }
    if (t <= Q8_GEMV_MAX_TOKENS) return q8::gemv_small_launch(w, n, k, qs, ds, y, t, s);
    if (t <= q8::kSlicedMaxTokens) return q8::gemv_sliced_launch(w, n, k, qs, ds, y, t, s);
    if (!gemm_tc_shape_ok(n, t, k)) return Q8_ERR_ARG;
    return q8::gemm_tc_launch(w, n, k, qs, ds, t, y, workspace, s);
}

extern "C" size_t q8_0_gemm_prepared_weights_bytes(int64_t n, int64_t k)
{
    if (n < 1 || k <= 0 || (k % 32) != 0 || (k / 32) % 8 != 0 || !gemm_tc_shape_ok(n, 1, k)) return 0;
    return q8::gemm_prepared_weights_bytes(n, k);
}

extern "C" int q8_0_gemm_prepare_weights(const void *w, int64_t n, int64_t k, void *wprep, size_t wprep_bytes,
                                         void *stream)
{
    if (!w || !wprep || n < 1 || k <= 0 || (k % 32) != 0 || (k / 32) % 8 != 0 || !gemm_tc_shape_ok(n, 1, k))
        return Q8_ERR_ARG;
    if (wprep_bytes < q8_0_gemm_prepared_weights_bytes(n, k)) return Q8_ERR_ARG;
    if (!q8::aligned16(w) || !q8::aligned16(wprep)) return Q8_ERR_ALIGN;
    if (!q8::device_is_sm103()) return Q8_ERR_DEVICE;
    return q8::gemm_prepare_weights_launch(w, n, k, wprep, static_cast<cudaStream_t>(stream));
}

extern "C" size_t q8_0_gemm_prepared_workspace_bytes(int64_t n, int64_t t, int64_t k)
{
    if (n < 1 || t <= q8::kSlicedMaxTokens || k <= 0 || (k % 32) != 0 || (k / 32) % 8 != 0) return 0;
    return q8::gemm_prepared_workspace_bytes(n, t, k);
}

extern "C" int q8_0_gemm_prepared(const void *w, const void *wprep, int64_t n, int64_t k, const int8_t *qs,
                                  const uint32_t *ds, int64_t t, int64_t rows_pad, float *y, void *workspace,
                                  size_t workspace_bytes, void *stream)
{
    if (!qs || !ds || !y || n < 1 || t < 1 || k <= 0 || (k % 32) != 0 || rows_pad < t) return Q8_ERR_ARG;
    const bool tc = (k / 32) % 8 == 0 && t > q8::kSlicedMaxTokens;  // the tcgen05 path reads wprep, the rest w
    if (tc ? !wprep : !w) return Q8_ERR_ARG;
    if (!q8::aligned16(qs) || !q8::aligned16(ds) || !q8::aligned16(y) ||
        (tc ? !q8::aligned16(wprep) : !q8::aligned16(w)))
        return Q8_ERR_ALIGN;
    if (!tc) return q8_0_gemm(w, n, k, qs, ds, t, rows_pad, y, nullptr, 0, stream);
    const size_t need = q8_0_gemm_prepared_workspace_bytes(n, t, k);
    if (!workspace || workspace_bytes < need) return Q8_ERR_ARG;
    if (!q8::aligned16(workspace)) return Q8_ERR_ALIGN;
    if (!gemm_tc_shape_ok(n, t, k)) return Q8_ERR_ARG;
    if (!q8::device_is_sm103()) return Q8_ERR_DEVICE;
    return q8::gemm_tc_prepared_launch(wprep, n, k, qs, ds, t, y, workspace, static_cast<cudaStream_t>(stream));
}

extern "C" int q8_0_gemm_mma(const void *w, int64_t n, int64_t k, const int8_t *qs, const uint32_t *ds, int64_t t,
                             int64_t rows_pad, float *y, void *stream)
{
    if (!w || !qs || !ds || !y || n < 1 || t < 1 || k <= 0 || (k % 32) != 0 || rows_pad < t) return Q8_ERR_ARG;
    if ((k / 32) % 8 != 0 || t > int64_t(65535) * 64) return Q8_ERR_ARG;
    if (!q8::aligned16(w) || !q8::aligned16(qs) || !q8::aligned16(ds) || !q8::aligned16(y)) return Q8_ERR_ALIGN;
    if (!q8::device_is_sm103()) return Q8_ERR_DEVICE;
    return q8::gemm_mma_launch(w, n, k, qs, ds, t, y, static_cast<cudaStream_t>(stream));
}
