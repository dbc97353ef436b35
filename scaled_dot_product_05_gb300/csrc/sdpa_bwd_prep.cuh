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
// D / 8 16-byte loads, one per lane of a group of D / 8 lanes.
constexpr int kDeltaThreads = 256;
template <int D>
__host__ __device__ constexpr int delta_rows_per_block()
{
    return kDeltaThreads / (D / 8);
}

// Delta_i = dO_i . O_i (fp32) for every row (b, i, hq), read in memory order
// ([B][Sq][Hq][D], 16-bit) and written to the [B][Hq][Sq] layout.
template <int D, bool kBF16>
__global__ void __launch_bounds__(kDeltaThreads) bwd_delta_kernel(const void* O, const void* dO, float* delta,
                                                                  int B, int Hq, int Sq)
{
    constexpr int kLanes = D / 8;
    const int64_t rows = (int64_t)B * Sq * Hq;
    const int64_t row = (int64_t)blockIdx.x * delta_rows_per_block<D>() + threadIdx.x / kLanes;
    const int c = threadIdx.x % kLanes;
    float acc = 0.f;
    if (row < rows) {
        const uint4 o = reinterpret_cast<const uint4*>(O)[row * kLanes + c];
        const uint4 g = reinterpret_cast<const uint4*>(dO)[row * kLanes + c];
        const uint32_t ov[4] = {o.x, o.y, o.z, o.w}, gv[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float2 of, gf;
            if constexpr (kBF16) {
                of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ov[k]));
                gf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gv[k]));
            } else {
                of = __half22float2(*reinterpret_cast<const __half2*>(&ov[k]));
                gf = __half22float2(*reinterpret_cast<const __half2*>(&gv[k]));
            }
            acc = fmaf(of.x, gf.x, acc);
            acc = fmaf(of.y, gf.y, acc);
        }
    }
    // every lane takes part in the group's sum
#pragma unroll
    for (int s = kLanes / 2; s > 0; s >>= 1)
        acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (row < rows && c == 0) {
        const int hq = (int)(row % Hq);
        const int64_t bi = row / Hq;
        const int i = (int)(bi % Sq);
        const int b = (int)(bi / Sq);
        delta[((int64_t)b * Hq + hq) * Sq + i] = acc;
    }
}

// dQ (16-bit, [B][Sq][Hq][D]) from the fp32 accumulator, 4 elements a thread.
template <bool kBF16>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float* acc, void* dQ, int64_t n)
{
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
    if (i >= n)
        return;
    const float4 v = *reinterpret_cast<const float4*>(acc + i);
    uint2 out;
    out.x = pack2<kBF16>(v.x, v.y);
    out.y = pack2<kBF16>(v.z, v.w);
    *reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(dQ) + i) = out;
}

}  // namespace bwd
}  // namespace sdpa
