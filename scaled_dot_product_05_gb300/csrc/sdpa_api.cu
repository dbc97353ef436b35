// sdpa_api.cu -- C ABI of the attention forward pass (declared in
// include/sdpa.h): argument checks, TMA tensor-map encoding and the launch.
//
// Every check runs before the first CUDA call, so a rejected call enqueues
// nothing.  Nothing here allocates device memory.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>
#include <utility>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/sdpa.h"
#include "sdpa_kernel.cuh"
#include "sdpa_bwd.cuh"
#include "sdpa_bwd_prep.cuh"
#include "sdpa_bwd_fp8.cuh"

namespace {

thread_local int t_last_cuda_error = 0;

// Scratch of sdpa_fwd_decode_noalloc: a file-scope device array (one instance
// per device, allocated with the module, never by a call; every process that
// loads the library holds these 32 MiB on each device it uses, whichever entry
// points it calls).  A split plan
// needs at most rows * splits * (D + 1) * 4 bytes with B * Hkv * pairs *
// splits <= #SMs, i.e. #SMs * 256 * 129 * 4 bytes (about 20 MB on 152 SMs);
// larger plans are rejected.  Nothing in it needs to start at zero: every
// slot the merge reads is written earlier in the same call.  Calls that use
// it must not overlap in time (same stream, or otherwise ordered).
constexpr size_t kDecodeScratchBytes = size_t(32) << 20;
static __device__ __align__(256) float g_decode_scratch[kDecodeScratchBytes / sizeof(float)];

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
    // this device's instance of g_decode_scratch, looked up once
    std::once_flag scratch_once;
    cudaError_t scratch_err = cudaSuccess;
    void* scratch = nullptr;
};
DeviceState g_dev[kMaxDevices];

template <int D, int KIND, bool kPacked = false, int QT = 2>
cudaError_t set_attrs()
{
    return cudaFuncSetAttribute(sdpa::sdpa_fwd_kernel<D, KIND, kPacked, QT>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, sdpa::Layout<D, KIND, QT>::kSmemBytes);
}

template <int D, int KIND>
cudaError_t set_bwd_attrs()
{
    return cudaFuncSetAttribute(sdpa::bwd::sdpa_bwd_kernel<D, KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                sdpa::bwd::BwdLayout<D>::kSmemBytes);
}

template <int D>
cudaError_t set_bwd8_attrs()
{
    return cudaFuncSetAttribute(sdpa::bwd8::sdpa_bwd_fp8_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                sdpa::bwd8::Layout<D>::kSmemBytes);
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
        cudaError_t es[] = {set_attrs<32, sdpa::kBF16, false, 1>(), set_attrs<32, sdpa::kFP16, false, 1>(),
                            set_attrs<64, sdpa::kBF16, false, 1>(), set_attrs<64, sdpa::kFP16, false, 1>(),
                            set_attrs<32, sdpa::kBF16>(),        set_attrs<32, sdpa::kFP16>(),
                            set_attrs<64, sdpa::kBF16>(),        set_attrs<64, sdpa::kFP16>(),
                            set_attrs<64, sdpa::kE4M3>(),        set_attrs<128, sdpa::kBF16>(),
                            set_attrs<128, sdpa::kFP16>(),       set_attrs<128, sdpa::kE4M3>(),
                            set_attrs<32, sdpa::kBF16, true>(),  set_attrs<32, sdpa::kFP16, true>(),
                            set_attrs<64, sdpa::kBF16, true>(),  set_attrs<64, sdpa::kFP16, true>(),
                            set_attrs<128, sdpa::kBF16, true>(), set_attrs<128, sdpa::kFP16, true>(),
                            set_bwd_attrs<64, sdpa::kBF16>(),    set_bwd_attrs<64, sdpa::kFP16>(),
                            set_bwd_attrs<128, sdpa::kBF16>(),   set_bwd_attrs<128, sdpa::kFP16>(),
                            set_bwd8_attrs<64>(),                set_bwd8_attrs<128>()};
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

// Device address of the current device's g_decode_scratch.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current, as device_ready leaves it) and
// kept.
sdpa_status_t decode_scratch(int dev, void** out)
{
    DeviceState& st = g_dev[dev];
    std::call_once(st.scratch_once, [&] { st.scratch_err = cudaGetSymbolAddress(&st.scratch, g_decode_scratch); });
    if (st.scratch_err != cudaSuccess)
        return cuda_fail(st.scratch_err);
    *out = st.scratch;
    return SDPA_OK;
}

bool aligned16(const void* p)
{
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

bool overlaps(const void* a, long long na, const void* b, long long nb)
{
    const unsigned __int128 a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + (unsigned long long)nb && b0 < a0 + (unsigned long long)na;
}

struct Shape {
    int B, Hq, Hkv, Sq, Skv, D;
};

// Element strides of a [B][S][H][D] tensor (D contiguous).
struct Strides {
    long long b, s, h;
};

Strides contiguous_bshd(int S, int H, int D)
{
    return {static_cast<long long>(S) * H * D, static_cast<long long>(H) * D, D};
}

Strides resolve(const sdpa_layout_t* l, int S, int H, int D)
{
    return l ? Strides{l->batch, l->seq, l->head} : contiguous_bshd(S, H, D);
}

// Bytes from the first element to one past the last one of a B x S x H x D
// tensor with strides st (all strides > 0), or -1 past 2^62 bytes.
long long span_bytes(const Strides& st, int B, int S, int H, int D, int elem_bytes)
{
    const __int128 last = (__int128)(B - 1) * st.b + (__int128)(S - 1) * st.s + (__int128)(H - 1) * st.h + D;
    const __int128 bytes = last * elem_bytes;
    return bytes > ((__int128)1 << 62) ? -1 : static_cast<long long>(bytes);
}

// A stride the TMA engine and the 16-byte output stores accept: > 0, a
// multiple of 16 bytes, below 2^40 bytes.
bool stride_ok(long long st, int elem_bytes)
{
    if (st <= 0 || st > (1ll << 40) / elem_bytes)
        return false;
    return (st * elem_bytes) % 16 == 0;
}

bool strides_ok(const Strides& st, int elem_bytes)
{
    return stride_ok(st.b, elem_bytes) && stride_ok(st.s, elem_bytes) && stride_ok(st.h, elem_bytes);
}

// No two (b, s, h, d) of a B x S x H x D tensor share an address: with the
// dimensions of size > 1 sorted by stride, each stride reaches past the span
// of the smaller ones (D contiguous comes first).
bool injective(const Strides& st, int B, int S, int H, int D)
{
    long long dims[3][2] = {{st.b, B}, {st.s, S}, {st.h, H}};
    for (int i = 0; i < 3; ++i)                      // sort by stride
        for (int j = i + 1; j < 3; ++j)
            if (dims[j][0] < dims[i][0]) {
                std::swap(dims[i][0], dims[j][0]);
                std::swap(dims[i][1], dims[j][1]);
            }
    long long reach = D;                             // span of the dimensions so far
    for (int i = 0; i < 3; ++i) {
        if (dims[i][1] == 1)
            continue;
        if (dims[i][0] < reach)
            return false;
        reach = dims[i][0] * (dims[i][1] - 1) + reach;
    }
    return true;
}

bool aligned(const void* p, unsigned bytes)
{
    return (reinterpret_cast<uintptr_t>(p) & (bytes - 1)) == 0;
}

struct Args {
    const void *Q, *K, *V;
    void* O;
    float* lse;
    Shape s;
    Strides q, k, v, o;
};

// Checks shared by every entry point; no CUDA call.
sdpa_status_t check_common(const Args& a, int in_elem_bytes, int out_elem_bytes)
{
    const Shape& s = a.s;
    if (!a.Q || !a.K || !a.V || !a.O)
        return SDPA_ERR_NULL_PTR;
    if (!aligned16(a.Q) || !aligned16(a.K) || !aligned16(a.V) || !aligned16(a.O) || !aligned(a.lse, 4))
        return SDPA_ERR_MISALIGNED;
    if (s.B < 1 || s.Hq < 1 || s.Hkv < 1 || s.Sq < 1 || s.Skv < 1)
        return SDPA_ERR_BAD_SHAPE;
    if (s.Hq % s.Hkv != 0)
        return SDPA_ERR_HEADS;
    // D = 32 only for 16-bit elements: E4M3 rows would be 32 bytes
    if (s.D != 64 && s.D != 128 && !(s.D == 32 && in_elem_bytes == 2))
        return SDPA_ERR_HEAD_DIM;
    // the B * Hq * ceil(Sq / 128) work units (at most: units of one Q tile)
    // are counted in int
    const int64_t n_pairs = (static_cast<int64_t>(s.Sq) + sdpa::kBlockM - 1) / sdpa::kBlockM;
    if (static_cast<int64_t>(s.B) * s.Hq * n_pairs > INT32_MAX)
        return SDPA_ERR_BAD_SHAPE;
    if (!strides_ok(a.q, in_elem_bytes) || !strides_ok(a.k, in_elem_bytes) || !strides_ok(a.v, in_elem_bytes) ||
        !strides_ok(a.o, out_elem_bytes) || !injective(a.o, s.B, s.Sq, s.Hq, s.D))
        return SDPA_ERR_LAYOUT;
    const long long q_bytes = span_bytes(a.q, s.B, s.Sq, s.Hq, s.D, in_elem_bytes);
    const long long k_bytes = span_bytes(a.k, s.B, s.Skv, s.Hkv, s.D, in_elem_bytes);
    const long long v_bytes = span_bytes(a.v, s.B, s.Skv, s.Hkv, s.D, in_elem_bytes);
    const long long o_bytes = span_bytes(a.o, s.B, s.Sq, s.Hq, s.D, out_elem_bytes);
    if (q_bytes < 0 || k_bytes < 0 || v_bytes < 0 || o_bytes < 0)
        return SDPA_ERR_LAYOUT;
    if (overlaps(a.O, o_bytes, a.Q, q_bytes) || overlaps(a.O, o_bytes, a.K, k_bytes) ||
        overlaps(a.O, o_bytes, a.V, v_bytes))
        return SDPA_ERR_ALIAS;
    if (a.lse) {
        const long long l_bytes = static_cast<long long>(s.B) * s.Hq * s.Sq * static_cast<long long>(sizeof(float));
        if (overlaps(a.lse, l_bytes, a.Q, q_bytes) || overlaps(a.lse, l_bytes, a.K, k_bytes) ||
            overlaps(a.lse, l_bytes, a.V, v_bytes) || overlaps(a.lse, l_bytes, a.O, o_bytes))
            return SDPA_ERR_ALIAS;
    }
    return SDPA_OK;
}

bool valid_scale(float x)
{
    return std::isfinite(x) && x > 0.f;
}

// 4-D tensor map over a [B][S][H][D] tensor with element strides st: dims
// (innermost first) {D, H, S, B}, box {one swizzle chunk of the row (128
// bytes, or 64 when a row is 64 bytes), 1 head, 128 rows, 1 batch}, matching
// swizzle, zero fill out of bounds (ragged sequence tails).
bool encode_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, int D, int H, int S, int B,
                const Strides& st, int box_h, int box_s)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc)
        return false;
    const int row_bytes = D * elem_bytes;
    const int swz = row_bytes < 128 ? row_bytes : 128;
    const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)st.h * elem_bytes, (cuuint64_t)st.s * elem_bytes,
                                   (cuuint64_t)st.b * elem_bytes};
    const cuuint32_t box[4] = {(cuuint32_t)(swz / elem_bytes), (cuuint32_t)box_h, (cuuint32_t)box_s, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(map, dt, 4, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swz == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A tensor map depends only on these fields, so an encoded map can be reused
// whenever they repeat (repeated calls on the same buffers): a small
// per-thread cache, replaced round robin, saves the host-side encoding.
struct MapKey {
    const void* base;
    long long sb, ss, sh;
    int dt, elem_bytes, D, H, S, B, box_h, box_s;
};

// Tensor maps of earlier calls, per host thread.  Encoding one costs ~2 us of
// driver time, more than the rest of a small call; a call whose buffers,
// shapes and strides were seen before (a training or serving loop reuses its
// activation buffers, one model has a few maps per attention layer) finds its
// maps here.  Open addressing over kSlots entries, kProbes probes from the
// key's hash, replacement taking turns within the probe window.  The table
// (~0.8 MB) is allocated on a thread's first call.
struct MapCache {
    static constexpr uint32_t kSlots = 4096;     // a power of two
    static constexpr uint32_t kProbes = 8;
    struct Entry {
        CUtensorMap map;
        MapKey key;
        bool used;
    };
    std::vector<Entry> e = std::vector<Entry>(kSlots);
    uint32_t turn = 0;
};

thread_local MapCache t_maps;

// FNV-1a over the key's bytes (its padding is zeroed), folded
uint64_t map_key_hash(const MapKey& k)
{
    const unsigned char* b = reinterpret_cast<const unsigned char*>(&k);
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i < sizeof k; ++i) {
        h ^= b[i];
        h *= 1099511628211ull;
    }
    return h ^ (h >> 32);
}

// box_h x box_s (heads x rows) per copy: 1 x 128, or G x 128 / G for packed
// query tiles.
bool make_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem_bytes, int D, int H, int S, int B,
              const Strides& st, int box_h = 1, int box_s = sdpa::kBlockM)
{
    MapKey k;
    std::memset(&k, 0, sizeof k);                    // padding bytes take part in the comparison
    k.base = base;
    k.sb = st.b;
    k.ss = st.s;
    k.sh = st.h;
    k.dt = static_cast<int>(dt);
    k.elem_bytes = elem_bytes;
    k.D = D;
    k.H = H;
    k.S = S;
    k.B = B;
    k.box_h = box_h;
    k.box_s = box_s;
    MapCache& c = t_maps;
    const uint32_t h = static_cast<uint32_t>(map_key_hash(k));
    uint32_t free_slot = MapCache::kSlots;
    for (uint32_t i = 0; i < MapCache::kProbes; ++i) {
        MapCache::Entry& x = c.e[(h + i) & (MapCache::kSlots - 1)];
        if (!x.used) {
            if (free_slot == MapCache::kSlots)
                free_slot = (h + i) & (MapCache::kSlots - 1);
        } else if (std::memcmp(&x.key, &k, sizeof k) == 0) {
            *map = x.map;
            return true;
        }
    }
    if (!encode_map(map, base, dt, elem_bytes, D, H, S, B, st, box_h, box_s))
        return false;
    const uint32_t slot = free_slot != MapCache::kSlots
                              ? free_slot
                              : (h + c.turn++ % MapCache::kProbes) & (MapCache::kSlots - 1);
    MapCache::Entry& x = c.e[slot];
    std::memcpy(&x.key, &k, sizeof k);
    x.map = *map;
    x.used = true;
    return true;
}

// Launches `kernel`, with programmatic stream serialization when `pdl`: it
// may then start while the previous kernel in the stream finishes.  Every
// kernel launched here executes griddepcontrol.wait before touching global
// memory (a no-op in a plain launch), so it sees everything the previous
// kernel wrote and does not overwrite what that kernel still reads.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int D, int KIND, bool kPacked = false, int QT = 2>
cudaError_t launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                   const sdpa::Params& p, int sm_count, cudaStream_t stream)
{
    // persistent: one CTA per SM (all 512 TMEM columns), or two per SM with
    // one Q tile each (256 columns each)
    using R = sdpa::Roles<QT>;
    const long long slots = static_cast<long long>(sm_count) * R::kCtasPerSm;
    const unsigned grid = static_cast<unsigned>(p.n_units < slots ? p.n_units : slots);
    // the CTAs may start their prologue while the previous kernel finishes
    cudaError_t e = launch_pdl(true, sdpa::sdpa_fwd_kernel<D, KIND, kPacked, QT>, dim3(grid), dim3(R::kThreads),
                               sdpa::Layout<D, KIND, QT>::kSmemBytes, stream, tq, tk, tv, to, p);
    if constexpr (kPacked) {
        if (e == cudaSuccess && p.part_o) {
            // merge the key-range splits: one warp per output row
            const long long rows = static_cast<long long>(p.B) * p.Hq * p.Sq;
            sdpa::sdpa_combine_kernel<D, KIND != sdpa::kFP16>
                <<<static_cast<unsigned>((rows + 3) / 4), 128, 0, stream>>>(p);
            e = cudaGetLastError();
        }
    }
    return e;
}

// Q tiles per CTA of the standard forward pass.  One (two CTAs per SM, each
// loading its own K / V) for 16-bit kinds at D <= 64 when units of two Q
// tiles would fill at most two rounds of the SMs: there the finer units
// balance the causal work and one CTA's unit boundaries overlap the other's
// key tiles.  Else two (one CTA per SM, both tiles reading each K / V tile).
// Measured at D = 64, one against two: causal B=4 H=16 S=1024 (1.7 rounds)
// +6 %, the B=4 T=128 latency row +5 %; causal B=16 S=1024 (6.7 rounds) -6 %,
// causal S=2048..8192 -3 to -6 %, non-causal S=2048..16384 within 1 %.
int fwd_q_tiles(bool fp8, const Shape& s, int sm_count)
{
    if (fp8 || s.D > 64)
        return 2;
    const long long units2 =
        static_cast<long long>(s.B) * s.Hq * ((s.Sq + sdpa::kUnitRows - 1) / sdpa::kUnitRows);
    return units2 <= 2LL * sm_count ? 1 : 2;
}

sdpa::Params make_params(const Args& a, double score_scale, float out_scale, int causal, int unit_rows)
{
    const Shape& s = a.s;
    sdpa::Params p{};
    p.O = a.O;
    p.o_sb = a.o.b;
    p.o_ss = a.o.s;
    p.o_sh = a.o.h;
    p.lse = a.lse;
    p.B = s.B;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.Sq = s.Sq;
    p.Skv = s.Skv;
    p.group = s.Hq / s.Hkv;
    p.n_pairs = (s.Sq + unit_rows - 1) / unit_rows;
    p.n_units = s.B * s.Hq * p.n_pairs;
    p.n_ktiles = (s.Skv + sdpa::kBlockN - 1) / sdpa::kBlockN;
    p.causal = causal ? 1 : 0;
    p.scale_log2 = static_cast<float>(score_scale * 1.4426950408889634);   // exp(x) = exp2(x log2 e)
    p.out_scale = out_scale;
    return p;
}

template <int KIND>
cudaError_t launch_kind(int D, int qt, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const CUtensorMap& to, const sdpa::Params& p, int sm_count, cudaStream_t stream)
{
    // qt from fwd_q_tiles(), which also sized the units in p: one Q tile per
    // CTA only for 16-bit kinds at D <= 64
    if constexpr (KIND != sdpa::kE4M3) {
        if (qt == 1 && D == 32)
            return launch<32, KIND, false, 1>(tq, tk, tv, to, p, sm_count, stream);
        if (qt == 1 && D == 64)
            return launch<64, KIND, false, 1>(tq, tk, tv, to, p, sm_count, stream);
        if (qt == 1)
            return cudaErrorInvalidValue;       // never chosen at D = 128
        if (D == 32)
            return launch<32, KIND>(tq, tk, tv, to, p, sm_count, stream);
    } else if (D == 32 || qt != 2) {
        return cudaErrorInvalidValue;           // rejected by check_common / never chosen
    }
    return D == 64 ? launch<64, KIND>(tq, tk, tv, to, p, sm_count, stream)
                   : launch<128, KIND>(tq, tk, tv, to, p, sm_count, stream);
}

// The forward pass for already resolved arguments: checks, tensor maps,
// launch.  `descales` is null for 16-bit kinds.
sdpa_status_t run(const Args& a, float scale, const float* descales, int causal, sdpa_dtype_t dtype,
                  void* stream)
{
    const bool fp8 = dtype == SDPA_DTYPE_E4M3;
    const int in_bytes = fp8 ? 1 : 2;
    sdpa_status_t st = check_common(a, in_bytes, 2);
    if (st != SDPA_OK)
        return st;
    if (!valid_scale(scale))
        return SDPA_ERR_SCALE;
    double score_scale = scale;
    float out_scale = 1.f;
    if (fp8) {
        if (!valid_scale(descales[0]) || !valid_scale(descales[1]) || !valid_scale(descales[2]))
            return SDPA_ERR_SCALE;
        // the folded score scale must stay a finite, positive float
        score_scale = static_cast<double>(scale) * descales[0] * descales[1];
        const float c = static_cast<float>(score_scale * 1.4426950408889634);
        if (!(score_scale > 0.0) || !std::isfinite(c) || c == 0.f)
            return SDPA_ERR_SCALE;
        out_scale = descales[2];
    }

    int dev = 0, sm_count = 0;
    st = device_ready(&dev, &sm_count);
    if (st != SDPA_OK)
        return st;

    const Shape& s = a.s;
    const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                 : dtype == SDPA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                            : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    // O is written by TMA stores of 32 rows per softmax warp
    const CUtensorMapDataType dt_o = dtype == SDPA_DTYPE_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                              : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap tq, tk, tv, to;
    if (!make_map(&tq, a.Q, dt, in_bytes, s.D, s.Hq, s.Sq, s.B, a.q) ||
        !make_map(&tk, a.K, dt, in_bytes, s.D, s.Hkv, s.Skv, s.B, a.k) ||
        !make_map(&tv, a.V, dt, in_bytes, s.D, s.Hkv, s.Skv, s.B, a.v) ||
        !make_map(&to, a.O, dt_o, 2, s.D, s.Hq, s.Sq, s.B, a.o, 1, 32))
        return cuda_fail(cudaErrorInvalidValue);

    const int qt = fwd_q_tiles(fp8, s, sm_count);
    const sdpa::Params p = make_params(a, score_scale, out_scale, causal, qt * sdpa::kBlockM);
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const cudaError_t e = fp8 ? launch_kind<sdpa::kE4M3>(s.D, qt, tq, tk, tv, to, p, sm_count, cs)
                        : dtype == SDPA_DTYPE_BF16 ? launch_kind<sdpa::kBF16>(s.D, qt, tq, tk, tv, to, p, sm_count, cs)
                                                   : launch_kind<sdpa::kFP16>(s.D, qt, tq, tk, tv, to, p, sm_count, cs);
    if (e != cudaSuccess)
        return cuda_fail(e);
    return SDPA_OK;
}

// Packed (decode) pass plan: the G = Hq / Hkv query heads of a KV head are
// stacked into Q tiles (G must divide 128), and with a workspace the key
// range is split so that the units fill at most one wave of the SMs, each
// split at least 4 key tiles long.  The pass streams K and V from HBM: about
// a wave of units already saturates it, and more splits only add merge
// traffic (measured: 2 units per SM ran 10 % slower than 1).
struct DecodePlan {
    int n_pairs, n_splits, tiles_per_split;
    long long units;
    size_t workspace_bytes;          // 0 when there is one split
};

DecodePlan plan_decode(const Shape& s, int sm_count, bool split)
{
    DecodePlan d{};
    const int G = s.Hq / s.Hkv;
    const long long rows_packed = static_cast<long long>(s.Sq) * G;
    d.n_pairs = static_cast<int>((rows_packed + sdpa::kUnitRows - 1) / sdpa::kUnitRows);
    const long long base = static_cast<long long>(s.B) * s.Hkv * d.n_pairs;
    const int n_ktiles = (s.Skv + sdpa::kBlockN - 1) / sdpa::kBlockN;
    int splits = 1;
    if (split) {
        const long long want = sm_count / base;
        const int max_splits = n_ktiles / 4 > 1 ? n_ktiles / 4 : 1;
        splits = static_cast<int>(want < max_splits ? want : max_splits);
        if (splits < 1)
            splits = 1;
    }
    d.tiles_per_split = (n_ktiles + splits - 1) / splits;
    d.n_splits = (n_ktiles + d.tiles_per_split - 1) / d.tiles_per_split;
    d.units = base * d.n_splits;
    const long long rows = static_cast<long long>(s.B) * s.Hq * s.Sq;
    d.workspace_bytes = d.n_splits > 1 ? static_cast<size_t>(rows) * d.n_splits * (s.D + 1) * sizeof(float) : 0;
    return d;
}

sdpa_status_t run_decode(const Args& a, float scale, sdpa_dtype_t dtype, void* ws, size_t ws_bytes, void* stream)
{
    if (dtype != SDPA_DTYPE_BF16 && dtype != SDPA_DTYPE_FP16)
        return SDPA_ERR_DTYPE;
    sdpa_status_t st = check_common(a, 2, 2);
    if (st != SDPA_OK)
        return st;
    if (!valid_scale(scale))
        return SDPA_ERR_SCALE;
    const Shape& s = a.s;
    const int G = s.Hq / s.Hkv;
    if (sdpa::kBlockM % G != 0)
        return SDPA_ERR_HEADS;
    if (ws && !aligned16(ws))
        return SDPA_ERR_WORKSPACE;

    int dev = 0, sm_count = 0;
    st = device_ready(&dev, &sm_count);
    if (st != SDPA_OK)
        return st;
    const DecodePlan d = plan_decode(s, sm_count, ws != nullptr);
    if (d.units > INT32_MAX)
        return SDPA_ERR_BAD_SHAPE;
    if (d.workspace_bytes > ws_bytes)
        return SDPA_ERR_WORKSPACE;
    if (d.workspace_bytes) {
        const long long wb = static_cast<long long>(d.workspace_bytes);
        const long long q_bytes = span_bytes(a.q, s.B, s.Sq, s.Hq, s.D, 2);
        const long long k_bytes = span_bytes(a.k, s.B, s.Skv, s.Hkv, s.D, 2);
        const long long v_bytes = span_bytes(a.v, s.B, s.Skv, s.Hkv, s.D, 2);
        const long long o_bytes = span_bytes(a.o, s.B, s.Sq, s.Hq, s.D, 2);
        if (overlaps(ws, wb, a.Q, q_bytes) || overlaps(ws, wb, a.K, k_bytes) || overlaps(ws, wb, a.V, v_bytes) ||
            overlaps(ws, wb, a.O, o_bytes) ||
            (a.lse && overlaps(ws, wb, a.lse, static_cast<long long>(s.B) * s.Hq * s.Sq * 4)))
            return SDPA_ERR_ALIAS;
    }

    const CUtensorMapDataType dt =
        dtype == SDPA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUtensorMap tq, tk, tv;
    if (!make_map(&tq, a.Q, dt, 2, s.D, s.Hq, s.Sq, s.B, a.q, G, sdpa::kBlockM / G) ||
        !make_map(&tk, a.K, dt, 2, s.D, s.Hkv, s.Skv, s.B, a.k) ||
        !make_map(&tv, a.V, dt, 2, s.D, s.Hkv, s.Skv, s.B, a.v))
        return cuda_fail(cudaErrorInvalidValue);

    sdpa::Params p = make_params(a, scale, 1.f, 0, sdpa::kUnitRows);
    p.n_pairs = d.n_pairs;
    p.n_units = static_cast<int>(d.units);
    p.tiles_per_split = d.tiles_per_split;
    p.n_splits = d.n_splits;
    if (d.workspace_bytes) {
        const long long rows = static_cast<long long>(s.B) * s.Hq * s.Sq;
        p.part_o = static_cast<float*>(ws);
        p.part_lse = p.part_o + rows * d.n_splits * s.D;
    }
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    CUtensorMap unused;                  // packed mode writes O with plain stores
    std::memset(&unused, 0, sizeof unused);
    cudaError_t e;
    if (dtype == SDPA_DTYPE_BF16)
        e = s.D == 32 ? launch<32, sdpa::kBF16, true>(tq, tk, tv, unused, p, sm_count, cs)
          : s.D == 64 ? launch<64, sdpa::kBF16, true>(tq, tk, tv, unused, p, sm_count, cs)
                      : launch<128, sdpa::kBF16, true>(tq, tk, tv, unused, p, sm_count, cs);
    else
        e = s.D == 32 ? launch<32, sdpa::kFP16, true>(tq, tk, tv, unused, p, sm_count, cs)
          : s.D == 64 ? launch<64, sdpa::kFP16, true>(tq, tk, tv, unused, p, sm_count, cs)
                      : launch<128, sdpa::kFP16, true>(tq, tk, tv, unused, p, sm_count, cs);
    if (e != cudaSuccess)
        return cuda_fail(e);
    return SDPA_OK;
}

// Backward pass workspace: the fp32 dQ accumulator [B][Sq][Hq][D], then
// Delta [B][Hq][Sq].
size_t bwd_workspace(int B, int Hq, int Sq, int D)
{
    return static_cast<size_t>(B) * Sq * Hq * D * sizeof(float) + static_cast<size_t>(B) * Hq * Sq * sizeof(float);
}

// Whether a backward call launches its three kernels (Delta pass, main
// kernel, dQ conversion) with programmatic serialization: for short calls,
// of at most 64 (query tile, key tile) iterations per SM, whose kernels'
// launch latency and prologue are a visible share.  Measured against plain
// launches: causal MHA B=4 H=16 S=1024 D=64 (15 per SM) +10 %; causal GQA
// S=4096 D=128 (222 per SM) -3.5 %, so long calls launch plainly.
bool bwd_short_call(const Shape& s, bool causal, int sm_count)
{
    const long long n_qt = (s.Sq + sdpa::kBlockM - 1) / sdpa::kBlockM;
    const long long n_kt = (s.Skv + sdpa::kBlockN - 1) / sdpa::kBlockN;
    long long per_head = n_qt * n_kt;
    if (causal) {                    // query tile qt meets key tiles 0..qt
        per_head = 0;
        for (long long kt = 0; kt < n_kt; ++kt)
            per_head += n_qt > kt ? n_qt - kt : 0;
    }
    return static_cast<long long>(s.B) * s.Hq * per_head <= 64LL * sm_count;
}

template <int D, int KIND>
cudaError_t launch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const CUtensorMap& tdq, const sdpa::bwd::Params& p, const void* O, const void* dO, void* dQ,
                       bool pdl, cudaStream_t stream)
{
    constexpr bool kBF16 = (KIND == sdpa::kBF16);
    const long long rows = static_cast<long long>(p.B) * p.Hq * p.Sq;
    // Delta, and the dQ accumulator zeroed, in one pass
    constexpr int kRows = sdpa::bwd::delta_rows_per_block<D>();
    cudaError_t e = launch_pdl(pdl, sdpa::bwd::bwd_delta_kernel<D, kBF16>, dim3(static_cast<unsigned>((rows + kRows - 1) / kRows)),
                               dim3(sdpa::bwd::kDeltaThreads), 0, stream, O, dO, const_cast<float*>(p.delta), p.dq_acc,
                               p.B, p.Hq, p.Sq);
    if (e != cudaSuccess)
        return e;
    const unsigned grid = static_cast<unsigned>(static_cast<long long>(p.B) * p.Hkv * p.n_kt);
    if ((e = launch_pdl(pdl, sdpa::bwd::sdpa_bwd_kernel<D, KIND>, dim3(grid), dim3(sdpa::bwd::kThreads),
                        sdpa::bwd::BwdLayout<D>::kSmemBytes, stream, tq, tk, tv, tdo, tdq, p)) != cudaSuccess)
        return e;
    const long long n = rows * D;
    return launch_pdl(pdl, sdpa::bwd::bwd_dq_convert_kernel<kBF16>, dim3(static_cast<unsigned>((n / 8 + 255) / 256)),
                      dim3(256), 0, stream, static_cast<const float*>(p.dq_acc), dQ, n);
}

sdpa_status_t run_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                      void* dQ, void* dK, void* dV, const Shape& s, float scale, int causal, sdpa_dtype_t dtype,
                      void* ws, size_t ws_bytes, void* stream)
{
    if (dtype != SDPA_DTYPE_BF16 && dtype != SDPA_DTYPE_FP16)
        return SDPA_ERR_DTYPE;
    const Args fwd{Q, K, V, dQ, nullptr, s, contiguous_bshd(s.Sq, s.Hq, s.D), contiguous_bshd(s.Skv, s.Hkv, s.D),
                   contiguous_bshd(s.Skv, s.Hkv, s.D), contiguous_bshd(s.Sq, s.Hq, s.D)};
    if (!O || !dO || !LSE || !dK || !dV || !ws)
        return SDPA_ERR_NULL_PTR;
    sdpa_status_t st = check_common(fwd, 2, 2);      // Q, K, V, dQ: pointers, sizes, heads, dQ vs inputs
    if (st != SDPA_OK)
        return st;
    if (s.D != 64 && s.D != 128)
        return SDPA_ERR_HEAD_DIM;
    if (!aligned16(O) || !aligned16(dO) || !aligned16(dK) || !aligned16(dV) || !aligned16(ws) || !aligned(LSE, 4))
        return SDPA_ERR_MISALIGNED;
    if (!valid_scale(scale))
        return SDPA_ERR_SCALE;
    if (ws_bytes < bwd_workspace(s.B, s.Hq, s.Sq, s.D))
        return SDPA_ERR_WORKSPACE;
    const long long q_b = static_cast<long long>(s.B) * s.Sq * s.Hq * s.D * 2;
    const long long kv_b = static_cast<long long>(s.B) * s.Skv * s.Hkv * s.D * 2;
    const long long l_b = static_cast<long long>(s.B) * s.Hq * s.Sq * 4;
    const long long w_b = static_cast<long long>(bwd_workspace(s.B, s.Hq, s.Sq, s.D));
    // every written buffer (dQ, dK, dV, workspace) apart from every other buffer
    const void* bufs[10] = {Q, K, V, O, dO, LSE, dQ, dK, dV, ws};
    const long long lens[10] = {q_b, kv_b, kv_b, q_b, q_b, l_b, q_b, kv_b, kv_b, w_b};
    for (int w = 6; w < 10; ++w)
        for (int o = 0; o < 10; ++o)
            if (o != w && overlaps(bufs[w], lens[w], bufs[o], lens[o]))
                return SDPA_ERR_ALIAS;

    int dev = 0, sm_count = 0;
    st = device_ready(&dev, &sm_count);
    if (st != SDPA_OK)
        return st;
    const CUtensorMapDataType dt =
        dtype == SDPA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    // the fp32 dQ accumulator [B][Sq][Hq][D] at the start of the workspace
    // takes TMA reductions: boxes of 32 columns x 128 rows, 128-byte swizzle
    float* dq_acc = static_cast<float*>(ws);
    CUtensorMap tq, tk, tv, tdo, tdq;
    if (!make_map(&tq, Q, dt, 2, s.D, s.Hq, s.Sq, s.B, fwd.q) || !make_map(&tk, K, dt, 2, s.D, s.Hkv, s.Skv, s.B, fwd.k) ||
        !make_map(&tv, V, dt, 2, s.D, s.Hkv, s.Skv, s.B, fwd.v) ||
        !make_map(&tdo, dO, dt, 2, s.D, s.Hq, s.Sq, s.B, fwd.q) ||
        !make_map(&tdq, dq_acc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, s.D, s.Hq, s.Sq, s.B, fwd.q))
        return cuda_fail(cudaErrorInvalidValue);

    sdpa::bwd::Params p{};
    p.lse = LSE;
    p.dq_acc = dq_acc;
    p.delta = p.dq_acc + static_cast<long long>(s.B) * s.Sq * s.Hq * s.D;
    p.dK = dK;
    p.dV = dV;
    p.B = s.B;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.Sq = s.Sq;
    p.Skv = s.Skv;
    p.group = s.Hq / s.Hkv;
    p.n_qt = (s.Sq + sdpa::kBlockM - 1) / sdpa::kBlockM;
    p.n_kt = (s.Skv + sdpa::kBlockN - 1) / sdpa::kBlockN;
    p.causal = causal ? 1 : 0;
    p.scale = scale;
    p.scale_log2 = static_cast<float>(scale * 1.4426950408889634);
    if (static_cast<long long>(s.B) * s.Hkv * p.n_kt > INT32_MAX)
        return SDPA_ERR_BAD_SHAPE;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const bool pdl = bwd_short_call(s, causal != 0, sm_count);
    cudaError_t e;
    if (dtype == SDPA_DTYPE_BF16)
        e = s.D == 64 ? launch_bwd<64, sdpa::kBF16>(tq, tk, tv, tdo, tdq, p, O, dO, dQ, pdl, cs)
                      : launch_bwd<128, sdpa::kBF16>(tq, tk, tv, tdo, tdq, p, O, dO, dQ, pdl, cs);
    else
        e = s.D == 64 ? launch_bwd<64, sdpa::kFP16>(tq, tk, tv, tdo, tdq, p, O, dO, dQ, pdl, cs)
                      : launch_bwd<128, sdpa::kFP16>(tq, tk, tv, tdo, tdq, p, O, dO, dQ, pdl, cs);
    if (e != cudaSuccess)
        return cuda_fail(e);
    return SDPA_OK;
}

// FP8 backward workspace: the bf16 dQ accumulator [B][Sq][Hq][D], Delta
// [B][Hq][Sq] (fp32), then one 16-byte word for amax|dS| when the caller
// passes none.
size_t bwd8_dq_bytes(int B, int Hq, int Sq, int D)
{
    return static_cast<size_t>(B) * Sq * Hq * D * 2;
}

size_t bwd8_workspace(int B, int Hq, int Sq, int D)
{
    return bwd8_dq_bytes(B, Hq, Sq, D) + static_cast<size_t>(B) * Hq * Sq * sizeof(float) + 16;
}

template <int D>
cudaError_t launch_bwd8(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                        const CUtensorMap& tdq, const sdpa::bwd8::Params& p, const void* O, const void* dO8, void* dQ,
                        float dq_factor, bool pdl, cudaStream_t stream)
{
    const long long rows = static_cast<long long>(p.B) * p.Hq * p.Sq;
    // Delta, the dQ accumulator and amax zeroed, in one pass (two rows per
    // group of D / 16 lanes)
    constexpr int kRows = 2 * (256 / (D / 16));
    cudaError_t e = launch_pdl(pdl, sdpa::bwd8::bwd8_delta_kernel<D, true>, dim3(static_cast<unsigned>((rows + kRows - 1) / kRows)),
                               dim3(256), 0, stream, O, dO8, const_cast<float*>(p.delta), p.dq_acc, p.amax_ds, p.B, p.Hq,
                               p.Sq);
    if (e != cudaSuccess)
        return e;
    const unsigned grid = static_cast<unsigned>(static_cast<long long>(p.B) * p.Hkv * p.n_kt);
    if ((e = launch_pdl(pdl, sdpa::bwd8::sdpa_bwd_fp8_kernel<D>, dim3(grid), dim3(sdpa::bwd::kThreads),
                        sdpa::bwd8::Layout<D>::kSmemBytes, stream, tq, tk, tv, tdo, tdq, p)) != cudaSuccess)
        return e;
    const long long n = rows * D;
    return launch_pdl(pdl, sdpa::bwd8::bwd8_dq_convert_kernel, dim3(static_cast<unsigned>((n / 8 + 255) / 256)), dim3(256),
                      0, stream, static_cast<const uint16_t*>(p.dq_acc), dQ, n, dq_factor);
}

sdpa_status_t run_bwd_fp8(const void* Q8, const void* K8, const void* V8, const void* O, const void* dO8,
                          const float* LSE, void* dQ, void* dK, void* dV, const Shape& s, float scale, int causal,
                          float descale_q, float descale_k, float descale_v, float descale_do, float scale_ds,
                          float* amax_ds, void* ws, size_t ws_bytes, void* stream)
{
    // Q8, K8, V8, dO8 one byte an element; O, dQ, dK, dV bf16; all contiguous BSHD
    const Args fwd{Q8, K8, V8, dQ, nullptr, s, contiguous_bshd(s.Sq, s.Hq, s.D), contiguous_bshd(s.Skv, s.Hkv, s.D),
                   contiguous_bshd(s.Skv, s.Hkv, s.D), contiguous_bshd(s.Sq, s.Hq, s.D)};
    if (!O || !dO8 || !LSE || !dK || !dV || !ws)
        return SDPA_ERR_NULL_PTR;
    sdpa_status_t st = check_common(fwd, 1, 2);      // Q8, K8, V8, dQ: pointers, sizes, heads, dQ vs inputs
    if (st != SDPA_OK)
        return st;
    if (s.D != 64 && s.D != 128)
        return SDPA_ERR_HEAD_DIM;
    if (!aligned16(O) || !aligned16(dO8) || !aligned16(dK) || !aligned16(dV) || !aligned16(ws) || !aligned(LSE, 4) ||
        !aligned(amax_ds, 4))
        return SDPA_ERR_MISALIGNED;
    if (!valid_scale(scale) || !valid_scale(descale_q) || !valid_scale(descale_k) || !valid_scale(descale_v) ||
        !valid_scale(descale_do) || !valid_scale(scale_ds))
        return SDPA_ERR_SCALE;
    if (ws_bytes < bwd8_workspace(s.B, s.Hq, s.Sq, s.D))
        return SDPA_ERR_WORKSPACE;
    const long long q8_b = static_cast<long long>(s.B) * s.Sq * s.Hq * s.D;
    const long long kv8_b = static_cast<long long>(s.B) * s.Skv * s.Hkv * s.D;
    const long long q_b = 2 * q8_b, kv_b = 2 * kv8_b;
    const long long l_b = static_cast<long long>(s.B) * s.Hq * s.Sq * 4;
    const long long w_b = static_cast<long long>(bwd8_workspace(s.B, s.Hq, s.Sq, s.D));
    // every written buffer (dQ, dK, dV, workspace, amax) apart from every other buffer
    const void* bufs[11] = {Q8, K8, V8, O, dO8, LSE, dQ, dK, dV, ws, amax_ds};
    const long long lens[11] = {q8_b, kv8_b, kv8_b, q_b, q8_b, l_b, q_b, kv_b, kv_b, w_b, amax_ds ? 4 : 0};
    for (int w = 6; w < 11; ++w)
        for (int o = 0; o < 11; ++o)
            if (o != w && lens[w] > 0 && lens[o] > 0 && overlaps(bufs[w], lens[w], bufs[o], lens[o]))
                return SDPA_ERR_ALIAS;

    int dev = 0, sm_count = 0;
    st = device_ready(&dev, &sm_count);
    if (st != SDPA_OK)
        return st;
    uint16_t* dq_acc = static_cast<uint16_t*>(ws);
    CUtensorMap tq, tk, tv, tdo, tdq;
    const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (!make_map(&tq, Q8, u8, 1, s.D, s.Hq, s.Sq, s.B, fwd.q) || !make_map(&tk, K8, u8, 1, s.D, s.Hkv, s.Skv, s.B, fwd.k) ||
        !make_map(&tv, V8, u8, 1, s.D, s.Hkv, s.Skv, s.B, fwd.v) ||
        !make_map(&tdo, dO8, u8, 1, s.D, s.Hq, s.Sq, s.B, fwd.q) ||
        !make_map(&tdq, dq_acc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, s.D, s.Hq, s.Sq, s.B, fwd.q))
        return cuda_fail(cudaErrorInvalidValue);

    sdpa::bwd8::Params p{};
    p.lse = LSE;
    p.dq_acc = dq_acc;
    p.delta = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + bwd8_dq_bytes(s.B, s.Hq, s.Sq, s.D));
    p.amax_ds = amax_ds ? reinterpret_cast<unsigned int*>(amax_ds)
                        : reinterpret_cast<unsigned int*>(static_cast<uint8_t*>(ws) + bwd8_workspace(s.B, s.Hq, s.Sq, s.D) -
                                                          16);
    p.dK = dK;
    p.dV = dV;
    p.B = s.B;
    p.Hq = s.Hq;
    p.Hkv = s.Hkv;
    p.Sq = s.Sq;
    p.Skv = s.Skv;
    p.group = s.Hq / s.Hkv;
    p.n_qt = (s.Sq + sdpa::kBlockM - 1) / sdpa::kBlockM;
    p.n_kt = (s.Skv + sdpa::kBlockN - 1) / sdpa::kBlockN;
    p.causal = causal ? 1 : 0;
    p.c_s = static_cast<float>(static_cast<double>(scale) * descale_q * descale_k * 1.4426950408889634);
    p.dv = descale_v;
    p.ddo = descale_do;
    p.m_ds = descale_do * scale_ds;
    p.out_dv = descale_do / sdpa::bwd8::kPScale;
    p.out_dk = static_cast<float>(static_cast<double>(scale) * descale_q / scale_ds);
    const float dq_factor = static_cast<float>(static_cast<double>(scale) * descale_k / scale_ds);
    if (static_cast<long long>(s.B) * s.Hkv * p.n_kt > INT32_MAX)
        return SDPA_ERR_BAD_SHAPE;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const bool pdl = bwd_short_call(s, causal != 0, sm_count);
    const cudaError_t e = s.D == 64 ? launch_bwd8<64>(tq, tk, tv, tdo, tdq, p, O, dO8, dQ, dq_factor, pdl, cs)
                                    : launch_bwd8<128>(tq, tk, tv, tdo, tdq, p, O, dO8, dQ, dq_factor, pdl, cs);
    if (e != cudaSuccess)
        return cuda_fail(e);
    return SDPA_OK;
}

Args make_args(const void* Q, const void* K, const void* V, void* O, float* lse, int B, int Hq, int Hkv, int Sq,
               int Skv, int D, const sdpa_layout_t* ql, const sdpa_layout_t* kl, const sdpa_layout_t* vl,
               const sdpa_layout_t* ol)
{
    return Args{Q, K, V, O, lse, Shape{B, Hq, Hkv, Sq, Skv, D},
                resolve(ql, Sq, Hq, D), resolve(kl, Skv, Hkv, D), resolve(vl, Skv, Hkv, D), resolve(ol, Sq, Hq, D)};
}

}  // namespace

extern "C" {

sdpa_status_t sdpa_fwd(const void* Q, const void* K, const void* V, void* O, int B, int Hq, int Hkv, int Sq,
                       int Skv, int D, float scale, int causal, sdpa_dtype_t dtype, void* stream)
{
    return sdpa_fwd_ex(Q, K, V, O, nullptr, B, Hq, Hkv, Sq, Skv, D, nullptr, nullptr, nullptr, nullptr, scale,
                       causal, dtype, stream);
}

sdpa_status_t sdpa_fwd_ex(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int Hq, int Hkv,
                          int Sq, int Skv, int D, const sdpa_layout_t* q_layout, const sdpa_layout_t* k_layout,
                          const sdpa_layout_t* v_layout, const sdpa_layout_t* o_layout, float scale, int causal,
                          sdpa_dtype_t dtype, void* stream)
{
    if (dtype != SDPA_DTYPE_BF16 && dtype != SDPA_DTYPE_FP16)
        return SDPA_ERR_DTYPE;
    const Args a = make_args(Q, K, V, O, LSE, B, Hq, Hkv, Sq, Skv, D, q_layout, k_layout, v_layout, o_layout);
    return run(a, scale, nullptr, causal, dtype, stream);
}

sdpa_status_t sdpa_fwd_fp8(const void* Q, const void* K, const void* V, void* O, int B, int Hq, int Hkv, int Sq,
                           int Skv, int D, float scale, float descale_q, float descale_k, float descale_v,
                           int causal, void* stream)
{
    return sdpa_fwd_fp8_ex(Q, K, V, O, nullptr, B, Hq, Hkv, Sq, Skv, D, nullptr, nullptr, nullptr, nullptr, scale,
                           descale_q, descale_k, descale_v, causal, stream);
}

sdpa_status_t sdpa_fwd_fp8_ex(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int Hq,
                              int Hkv, int Sq, int Skv, int D, const sdpa_layout_t* q_layout,
                              const sdpa_layout_t* k_layout, const sdpa_layout_t* v_layout,
                              const sdpa_layout_t* o_layout, float scale, float descale_q, float descale_k,
                              float descale_v, int causal, void* stream)
{
    const Args a = make_args(Q, K, V, O, LSE, B, Hq, Hkv, Sq, Skv, D, q_layout, k_layout, v_layout, o_layout);
    const float descales[3] = {descale_q, descale_k, descale_v};
    return run(a, scale, descales, causal, SDPA_DTYPE_E4M3, stream);
}

sdpa_status_t sdpa_fwd_decode(const void* Q, const void* K, const void* V, void* O, float* LSE, int B, int Hq,
                              int Hkv, int Sq, int Skv, int D, const sdpa_layout_t* q_layout,
                              const sdpa_layout_t* k_layout, const sdpa_layout_t* v_layout,
                              const sdpa_layout_t* o_layout, float scale, sdpa_dtype_t dtype, void* workspace,
                              size_t workspace_bytes, void* stream)
{
    const Args a = make_args(Q, K, V, O, LSE, B, Hq, Hkv, Sq, Skv, D, q_layout, k_layout, v_layout, o_layout);
    return run_decode(a, scale, dtype, workspace, workspace_bytes, stream);
}

sdpa_status_t sdpa_fwd_decode_noalloc(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                                      int Hq, int Hkv, int Sq, int Skv, int D, const sdpa_layout_t* q_layout,
                                      const sdpa_layout_t* k_layout, const sdpa_layout_t* v_layout,
                                      const sdpa_layout_t* o_layout, float scale, sdpa_dtype_t dtype, void* stream)
{
    const Args a = make_args(Q, K, V, O, LSE, B, Hq, Hkv, Sq, Skv, D, q_layout, k_layout, v_layout, o_layout);
    // argument checks first, as for every entry point (run_decode repeats them)
    if (dtype != SDPA_DTYPE_BF16 && dtype != SDPA_DTYPE_FP16)
        return SDPA_ERR_DTYPE;
    const sdpa_status_t st = check_common(a, 2, 2);
    if (st != SDPA_OK)
        return st;
    if (!valid_scale(scale))
        return SDPA_ERR_SCALE;
    if (sdpa::kBlockM % (Hq / Hkv) != 0)
        return SDPA_ERR_HEADS;
    // the current device's instance of the library's scratch array
    int dev = 0, sm_count = 0;
    sdpa_status_t ds = device_ready(&dev, &sm_count);
    void* scratch = nullptr;
    if (ds == SDPA_OK)
        ds = decode_scratch(dev, &scratch);
    if (ds != SDPA_OK)
        return ds;
    return run_decode(a, scale, dtype, scratch, kDecodeScratchBytes, stream);
}

sdpa_status_t sdpa_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO, const float* LSE,
                       void* dQ, void* dK, void* dV, int B, int Hq, int Hkv, int Sq, int Skv, int D, float scale,
                       int causal, sdpa_dtype_t dtype, void* workspace, size_t workspace_bytes, void* stream)
{
    return run_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, Shape{B, Hq, Hkv, Sq, Skv, D}, scale, causal, dtype, workspace,
                   workspace_bytes, stream);
}

sdpa_status_t sdpa_bwd_fp8(const void* Q8, const void* K8, const void* V8, const void* O, const void* dO8,
                           const float* LSE, void* dQ, void* dK, void* dV, int B, int Hq, int Hkv, int Sq, int Skv,
                           int D, float scale, int causal, float descale_q, float descale_k, float descale_v,
                           float descale_do, float scale_ds, float* amax_ds, void* workspace, size_t workspace_bytes,
                           void* stream)
{
    return run_bwd_fp8(Q8, K8, V8, O, dO8, LSE, dQ, dK, dV, Shape{B, Hq, Hkv, Sq, Skv, D}, scale, causal, descale_q,
                       descale_k, descale_v, descale_do, scale_ds, amax_ds, workspace, workspace_bytes, stream);
}

size_t sdpa_bwd_fp8_workspace_bytes(int B, int Hq, int Sq, int D)
{
    if (B < 1 || Hq < 1 || Sq < 1 || (D != 64 && D != 128))
        return 0;
    return bwd8_workspace(B, Hq, Sq, D);
}

size_t sdpa_bwd_workspace_bytes(int B, int Hq, int Sq, int D)
{
    if (B < 1 || Hq < 1 || Sq < 1 || (D != 64 && D != 128))
        return 0;
    return bwd_workspace(B, Hq, Sq, D);
}

size_t sdpa_decode_workspace_bytes(int B, int Hq, int Hkv, int Sq, int Skv, int D)
{
    if (B < 1 || Hq < 1 || Hkv < 1 || Sq < 1 || Skv < 1 || Hq % Hkv != 0 || (D != 32 && D != 64 && D != 128))
        return 0;
    int dev = 0, sm_count = 0;
    if (device_ready(&dev, &sm_count) != SDPA_OK)
        return 0;
    return plan_decode(Shape{B, Hq, Hkv, Sq, Skv, D}, sm_count, true).workspace_bytes;
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
    case SDPA_ERR_LAYOUT: return "unusable strides";
    case SDPA_ERR_WORKSPACE: return "workspace too small or not 16-byte aligned";
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
    return 5;
}

#ifdef SDPA_WAIT_TEST
// Test build only (not declared in include/sdpa.h, not in the product
// library): sets the device wait limit in nanoseconds and the K-ring position
// (per CTA, counted from 0) whose copy the forward producer leaves out (-1:
// none).  With a position set, the waits that depend on that tile run out
// after `limit_ns`, the kernel records its code in the device error word and
// returns; the tests read the code through sdpa_device_error().
sdpa_status_t sdpa_test_set_wait(unsigned long long limit_ns, int withhold_k)
{
    const uint64_t lim = limit_ns;
    cudaError_t e = cudaMemcpyToSymbol(sdpa::g_test_wait_limit_ns, &lim, sizeof lim);
    if (e == cudaSuccess)
        e = cudaMemcpyToSymbol(sdpa::g_test_withhold_k, &withhold_k, sizeof withhold_k);
    return e == cudaSuccess ? SDPA_OK : cuda_fail(e);
}
#endif

}  // extern "C"
