// sdpa_bwd_prep.cuh -- the two small kernels around the backward pass:
// Delta_i = dO_i . O_i before it (the row term of dS = P * (dP - Delta) in
// section 1, "How attention works", of the codelab "Attention on GPU (cuDNN
// and TransformerEngine)", differentiated), and the conversion of the fp32 dQ
// accumulator to 16-bit after it.  Both are HBM-bound streams.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "sdpa_kernel.cuh"

namespace sdpa {
namespace bwd {

// Threads per Delta block, and rows per block: a row of D 16-bit values is
// D / 8 16-byte loads, one per lane of a group of D / 8 lanes; each group
// takes two rows, so that every lane has four loads in flight.
constexpr int kDeltaThreads = 256;
constexpr int kDeltaRowsPerGroup = 2;
template <int D>
__host__ __device__ constexpr int delta_rows_per_block()
{
    return kDeltaRowsPerGroup * (kDeltaThreads / (D / 8));
}

// Delta_i = dO_i . O_i (fp32) for every row (b, i, hq), read in memory order
// ([B][Sq][Hq][D], 16-bit) and written to the [B][Hq][Sq] layout.  The same
// pass zeroes the row's D fp32 of the dQ accumulator (also [B][Sq][Hq][D]),
// which the backward kernel then adds into: one launch instead of a memset
// and this kernel.
template <int D, bool kBF16>
__global__ void __launch_bounds__(kDeltaThreads) bwd_delta_kernel(const void* O, const void* dO, float* delta,
                                                                  float* dq_acc, int B, int Hq, int Sq)
{
    grid_dependency_wait();                       // launched with programmatic serialization
    grid_launch_dependents();
    constexpr int kLanes = D / 8;
    constexpr int kGroups = kDeltaThreads / kLanes;
    const int64_t rows = (int64_t)B * Sq * Hq;
    const int c = threadIdx.x % kLanes;
    int64_t row[kDeltaRowsPerGroup];
    uint4 o[kDeltaRowsPerGroup], g[kDeltaRowsPerGroup];
#pragma unroll
    for (int k = 0; k < kDeltaRowsPerGroup; ++k) {
        row[k] = (int64_t)blockIdx.x * delta_rows_per_block<D>() + k * kGroups + threadIdx.x / kLanes;
        if (row[k] < rows) {
            o[k] = reinterpret_cast<const uint4*>(O)[row[k] * kLanes + c];
            g[k] = reinterpret_cast<const uint4*>(dO)[row[k] * kLanes + c];
        }
    }
#pragma unroll
    for (int k = 0; k < kDeltaRowsPerGroup; ++k) {
        float acc = 0.f;
        if (row[k] < rows) {
            uint4* z = reinterpret_cast<uint4*>(dq_acc + row[k] * D + 8 * c);
            z[0] = make_uint4(0u, 0u, 0u, 0u);
            z[1] = make_uint4(0u, 0u, 0u, 0u);
            const uint32_t ov[4] = {o[k].x, o[k].y, o[k].z, o[k].w}, gv[4] = {g[k].x, g[k].y, g[k].z, g[k].w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float2 of, gf;
                if constexpr (kBF16) {
                    of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ov[e]));
                    gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv[e]));
                } else {
                    of = __half22float2(*reinterpret_cast<const __half2*>(&ov[e]));
                    gf = __half22float2(*reinterpret_cast<const __half2*>(&gv[e]));
                }
                acc = fmaf(of.x, gf.x, acc);
                acc = fmaf(of.y, gf.y, acc);
            }
        }
        // every lane takes part in the group's sum
#pragma unroll
        for (int s = kLanes / 2; s > 0; s >>= 1)
            acc += __shfl_xor_sync(0xffffffffu, acc, s);
        if (row[k] < rows && c == 0) {
            const int hq = (int)(row[k] % Hq);
            const int64_t bi = row[k] / Hq;
            const int i = (int)(bi % Sq);
            const int b = (int)(bi / Sq);
            delta[((int64_t)b * Hq + hq) * Sq + i] = acc;
        }
    }
}

// dQ (16-bit, [B][Sq][Hq][D]) from the fp32 accumulator, 8 elements a thread
// (n is a multiple of 8: D is 64 or 128).
template <bool kBF16>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float* acc, void* dQ, int64_t n)
{
    grid_dependency_wait();                       // launched with programmatic serialization
    grid_launch_dependents();
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
    if (i >= n)
        return;
    const float4 a = *reinterpret_cast<const float4*>(acc + i);
    const float4 b = *reinterpret_cast<const float4*>(acc + i + 4);
    *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(dQ) + i) =
        make_uint4(pack2<kBF16>(a.x, a.y), pack2<kBF16>(a.z, a.w), pack2<kBF16>(b.x, b.y), pack2<kBF16>(b.z, b.w));
}

}  // namespace bwd
}  // namespace sdpa
