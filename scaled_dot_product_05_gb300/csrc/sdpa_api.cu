// sdpa_api.cu -- C ABI of the attention forward pass (declared in
// include/sdpa.h): argument checks, TMA tensor-map encoding and the launch.
//
// Every check runs before the first CUDA call, so a rejected call enqueues
// nothing.  Nothing here allocates device memory.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/sdpa.h"
#include "sdpa_kernel.cuh"

namespace {

thread_local int t_last_cuda_error = 0;

sdpa_status_t cuda_fail(cudaError_t e)
{
    t_last_cuda_error = static_cast<int>(e);
    return SDPA_ERR_CUDA;
}

constexpr int kMaxDevices = 64;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Per-device one-time state: architecture check and kernel attributes.
struct DeviceState {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    bool arch_ok = false;
    int sm_count = 0;
};
DeviceState g_dev[kMaxDevices];

template <int D, int KIND>
cudaError_t set_attrs()
{
    return cudaFuncSetAttribute(sdpa::sdpa_fwd_kernel<D, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                sdpa::Layout<D, KIND>::kSmemBytes);
}

sdpa_status_t device_ready(int* dev_out, int* sm_count)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return cuda_fail(e);
    if (dev < 0 || dev >= kMaxDevices)
        return SDPA_ERR_ARCH;
    DeviceState& st = g_dev[dev];
    std::call_once(st.once, [&] {
        int major = 0, minor = 0;
        cudaError_t e1 = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaError_t e2 = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e1 != cudaSuccess || e2 != cudaSuccess) {
            st.err = e1 != cudaSuccess ? e1 : e2;
            return;
        }
        st.arch_ok = (major == 10 && minor == 3);
        if (!st.arch_ok)
            return;
        cudaError_t e3 = cudaDeviceGetAttribute(&st.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e3 != cudaSuccess) {
            st.err = e3;
            return;
        }
        cudaError_t es[] = {set_attrs<64, sdpa::kBF16>(),  set_attrs<64, sdpa::kFP16>(),
                            set_attrs<64, sdpa::kE4M3>(),  set_attrs<128, sdpa::kBF16>(),
                            set_attrs<128, sdpa::kFP16>(), set_attrs<128, sdpa::kE4M3>()};
        for (cudaError_t x : es)
            if (x != cudaSuccess && st.err == cudaSuccess)
                st.err = x;
    });
    if (st.err != cudaSuccess)
        return cuda_fail(st.err);
    if (!st.arch_ok)
        return SDPA_ERR_ARCH;
    *dev_out = dev;
    *sm_count = st.sm_count;
    return SDPA_OK;
}

bool aligned16(const void* p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb)
{
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

struct Shape {
    int B, Hq, Hkv, Sq, Skv, D;
};

// Checks shared by both entry points; no CUDA call.
sdpa_status_t check_common(const void* Q, const void* K, const void* V, const void* O, const Shape& s,
                           int in_elem_bytes, int out_elem_bytes)
{
    if (!Q || !K || !V || !O)
        return SDPA_ERR_NULL_PTR;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O))
        return SDPA_ERR_MISALIGNED;
    if (s.B < 1 || s.Hq < 1 || s.Hkv < 1 || s.Sq < 1 || s.Skv < 1)
        return SDPA_ERR_BAD_SHAPE;
    if (s.Hq % s.Hkv != 0)
        return SDPA_ERR_HEADS;
    if (s.D != 64 && s.D != 128)
        return SDPA_ERR_HEAD_DIM;
    // the B * Hq * ceil(Sq / 256) work units are counted in int
    const int64_t n_pairs = (static_cast<int64_t>(s.Sq) + sdpa::kUnitRows - 1) / sdpa::kUnitRows;
    if (static_cast<int64_t>(s.B) * s.Hq * n_pairs > INT32_MAX)
        return SDPA_ERR_BAD_SHAPE;
    const size_t nq = static_cast<size_t>(s.B) * s.Sq * s.Hq * s.D;
    const size_t nkv = static_cast<size_t>(s.B) * s.Skv * s.Hkv * s.D;
    const size_t o_bytes = nq * out_elem_bytes;
    if (overlaps(O, o_bytes, Q, nq * in_elem_bytes) || overlaps(O, o_bytes, K, nkv * in_elem_bytes) ||
        overlaps(O, o_bytes, V, nkv * in_elem_bytes))
        return SDPA_ERR_ALIAS;
    return SDPA_OK;
}

bool valid_scale(float x)
{
    return std::isfinite(x) && x > 0.f;
}

// 4-D tensor map over a [B][S][H][D] array: dims (innermost first) {D, H, S, B},
// box {one swizzle chunk of the row (128 bytes, or 64 when a row is 64 bytes),
// 1 head, 128 rows, 1 batch}, matching swizzle, zero fill out of bounds
// (ragged sequence tails).
bool make_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, int D, int H, int S, int B)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const int row_bytes = D * elem_bytes;
    const int swz = row_bytes < 128 ? row_bytes : 128;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)D * elem_bytes, (cuuint64_t)H * D * elem_bytes,
                                   (cuuint64_t)S * H * D * elem_bytes};
    const cuuint32_t box[4] = {(cuuint32_t)(swz / elem_bytes), 1, (cuuint32_t)sdpa::kBlockM, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swz == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int KIND>
cudaError_t launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const sdpa::Params& p,
                   int sm_count, cudaStream_t stream)
{
    // persistent: one CTA per SM (each takes all 512 TMEM columns)
    const unsigned grid = static_cast<unsigned>(p.n_units < sm_count ? p.n_units : sm_count);
    sdpa::sdpa_fwd_kernel<D, KIND><<<grid, sdpa::kThreads, sdpa::Layout<D, KIND>::kSmemBytes, stream>>>(tq, tk, tv,
                                                                                                          p);
    return cudaGetLastError();
}

sdpa::Params make_params(void* O, const Shape& s, double score_scale, float out_scale, int causal)
{
    sdpa::Params p{};
    p.O = O;
    p.B = s.B;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.Sq = s.Sq;
    p.Skv = s.Skv;
    p.group = s.Hq / s.Hkv;
    p.n_pairs = (s.Sq + sdpa::kUnitRows - 1) / sdpa::kUnitRows;
    p.n_units = s.B * s.Hq * p.n_pairs;
    p.n_ktiles = (s.Skv + sdpa::kBlockN - 1) / sdpa::kBlockN;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = static_cast<float>(score_scale * 1.4426950408889634);   // exp(x) = exp2(x log2 e)
    p.out_scale = out_scale;
    return p;
}

template <int KIND>
cudaError_t launch_kind(int D, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const sdpa::Params& p, int sm_count, cudaStream_t stream)
{
    return D == 64 ? launch<64, KIND>(tq, tk, tv, p, sm_count, stream)
                   : launch<128, KIND>(tq, tk, tv, p, sm_count, stream);
}

}  // namespace

extern "C" {

sdpa_status_t sdpa_fwd(const void* Q, const void* K, const void* V, void* O, int B, int Hq, int Hkv, int Sq,
                       int Skv, int D, float scale, int causal, sdpa_dtype_t dtype, void* stream)
{
    if (dtype != SDPA_DTYPE_BF16 && dtype != SDPA_DTYPE_FP16)
        return SDPA_ERR_DTYPE;
    const Shape s{B, Hq, Hkv, Sq, Skv, D};
    sdpa_status_t st = check_common(Q, K, V, O, s, 2, 2);
    if (st != SDPA_OK)
        return st;
    if (!valid_scale(scale))
        return SDPA_ERR_SCALE;

    int dev = 0, sm_count = 0;
    st = device_ready(&dev, &sm_count);
    if (st != SDPA_OK)
        return st;

    const CUtensorMapDataType dt =
        dtype == SDPA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tq, tk, tv;
    if (!make_map(&tq, Q, dt, 2, D, Hq, Sq, B) || !make_map(&tk, K, dt, 2, D, Hkv, Skv, B) ||
        !make_map(&tv, V, dt, 2, D, Hkv, Skv, B))
        return cuda_fail(cudaErrorInvalidValue);

    const sdpa::Params p = make_params(O, s, scale, 1.f, causal);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const cudaError_t e = dtype == SDPA_DTYPE_BF16 ? launch_kind<sdpa::kBF16>(D, tq, tk, tv, p, sm_count, cs)
                                                   : launch_kind<sdpa::kFP16>(D, tq, tk, tv, p, sm_count, cs);
    if (e != cudaSuccess)
        return cuda_fail(e);
    return SDPA_OK;
}

sdpa_status_t sdpa_fwd_fp8(const void* Q, const void* K, const void* V, void* O, int B, int Hq, int Hkv, int Sq,
                           int Skv, int D, float scale, float descale_q, float descale_k, float descale_v,
                           int causal, void* stream)
{
    const Shape s{B, Hq, Hkv, Sq, Skv, D};
    sdpa_status_t st = check_common(Q, K, V, O, s, 1, 2);
    if (st != SDPA_OK)
        return st;
    if (!valid_scale(scale) || !valid_scale(descale_q) || !valid_scale(descale_k) || !valid_scale(descale_v))
        return SDPA_ERR_SCALE;
    // the folded score scale must stay a finite, positive float
    const double score_scale = static_cast<double>(scale) * descale_q * descale_k;
    if (!(score_scale > 0.0) || !std::isfinite(static_cast<float>(score_scale * 1.4426950408889634)) ||
        static_cast<float>(score_scale * 1.4426950408889634) == 0.f)
        return SDPA_ERR_SCALE;

    int dev = 0, sm_count = 0;
    st = device_ready(&dev, &sm_count);
    if (st != SDPA_OK)
        return st;

    CUtensorMap tq, tk, tv;
    const CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (!make_map(&tq, Q, dt, 1, D, Hq, Sq, B) || !make_map(&tk, K, dt, 1, D, Hkv, Skv, B) ||
        !make_map(&tv, V, dt, 1, D, Hkv, Skv, B))
        return cuda_fail(cudaErrorInvalidValue);

    const sdpa::Params p = make_params(O, s, score_scale, descale_v, causal);
    const cudaError_t e = launch_kind<sdpa::kE4M3>(D, tq, tk, tv, p, sm_count, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e);
    return SDPA_OK;
}

const char* sdpa_status_string(sdpa_status_t status)
{
    switch (status) {
    case SDPA_OK: return "ok";
    case SDPA_ERR_NULL_PTR: return "null pointer";
    case SDPA_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case SDPA_ERR_BAD_SHAPE: return "size out of range";
    case SDPA_ERR_HEADS: return "Hq is not a multiple of Hkv";
    case SDPA_ERR_HEAD_DIM: return "head dimension must be 64 or 128";
    case SDPA_ERR_DTYPE: return "unsupported dtype for this entry point";
    case SDPA_ERR_SCALE: return "scale / descale must be finite and > 0";
    case SDPA_ERR_ARCH: return "device is not compute capability 10.3 (GB300)";
    case SDPA_ERR_ALIAS: return "output overlaps an input";
    case SDPA_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

int sdpa_last_cuda_error(void)
{
    return t_last_cuda_error;
}

sdpa_status_t sdpa_device_error(unsigned int* code)
{
    if (!code)
        return SDPA_ERR_NULL_PTR;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return cuda_fail(e);
    unsigned int v = 0;
    e = cudaMemcpyFromSymbol(&v, sdpa::g_sdpa_error, sizeof v);
    if (e != cudaSuccess)
        return cuda_fail(e);
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(sdpa::g_sdpa_error, &zero, sizeof zero);
    if (e != cudaSuccess)
        return cuda_fail(e);
    *code = v;
    return SDPA_OK;
}

int sdpa_abi_version(void)
{
    return 1;
}

}  // extern "C"
