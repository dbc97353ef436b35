// sdpa_bwd_fp8.cuh -- FP8 backward pass of the attention forward pass, for
// sm_103a.
//
// The codelab "Attention on GPU (cuDNN and TransformerEngine)" trains in FP8
// with E4M3 tensors in the forward pass and E5M2 for the backward pass (section
// 10, "FP8": the hybrid format, delayed per-tensor scaling).  This kernel takes
// E4M3 Q, K, V and an E5M2 upstream gradient dO, each with its per-tensor
// descale (value = code * descale), the 16-bit O and the fp32 LSE of the
// forward pass, and runs all five GEMMs of the backward pass on the FP8 tensor
// cores (tcgen05 kind::f8f6f4, fp32 accumulators):
//     S^T  = K Q^T             E4M3 x E4M3
//     dP^T = V dO^T            E4M3 x E5M2
//     dV  += P8^T dO           E4M3 x E5M2   P8 = e4m3(P * 448), P <= 1
//     dK  += dS8^T Q           E5M2 x E4M3   dS8 = e5m2(dS * scale_ds)
//     dQ_part = dS8 K          E5M2 x E4M3
// with dS = P * (dP - Delta) formed in fp32 from P before its rounding.  The
// caller's scale_ds is the delayed scale of dS (the recipe's amax history);
// the kernel reports amax|dS| of this call for the next one.  The descales and
// 1/448, 1/scale_ds are folded into the epilogues; dQ, dK, dV are bf16.
//
// The structure follows the 16-bit kernel in sdpa_bwd.cuh (one CTA per batch,
// KV head and 128-key tile, dK and dV in TMEM over the query tiles of the
// group, longest first), with 8-bit operand tiles: P^T and dS^T go to shared
// memory for SS MMAs (keys x 128 queries, one 128-byte swizzled row per key),
// and dQ_part is staged in a buffer of its own (128 x D bf16), which 8-bit
// tiles leave room for, and added into a bf16 accumulator in global memory.
#pragma once

#include <cstdint>
#include <cuda.h>

#include "ptx.cuh"
#include "sdpa_bwd.cuh"
#include "sdpa_kernel.cuh"

namespace sdpa {
namespace bwd8 {

using bwd::kThreads;
using bwd::kProducerWarp;
using bwd::kMmaWarp;
using bwd::kReduceWarp;
using bwd::kStatsWarp;
using bwd::kSoftmaxWarp0;
using bwd::kDqWarp0;
using bwd::kRegsLow;
using bwd::kRegsSoftmax;
using bwd::kRegsDq;
using bwd::kLog2e;
using bwd::kSliceBytes;

constexpr unsigned int kErrBwd8Wait = 0x500;  // + barrier id: an FP8 backward wait timed out
constexpr float kPScale = 448.f;              // P in (0, 1] -> E4M3 codes up to 448

struct Params {
    const float* lse;                // [B][Hq][Sq] natural-log LSE of the forward pass
    const float* delta;              // [B][Hq][Sq] sum_d dO8 O (dO as codes)
    uint16_t* dq_acc;                // [B][Sq][Hq][D] bf16, zero on entry (see the reducer)
    void* dK;                        // [B][Skv][Hkv][D] bf16
    void* dV;
    unsigned int* amax_ds;           // max |dS| of this call, as fp32 bits (atomic max)
    int B, Hq, Hkv, Sq, Skv;
    int group;
    int n_qt, n_kt;
    int causal;
    float c_s;                       // scale * dq * dk * log2(e): S^T codes -> exp2 argument
    float dv;                        // descale of V (dP = ddo * dv * codes)
    float ddo;                       // descale of dO
    float m_ds;                      // ddo * scale_ds: (P (dv dP8 - Delta8)) -> E5M2 argument
    float out_dv;                    // ddo / 448
    float out_dk;                    // scale * dq / scale_ds
};

struct Barriers {
    uint64_t kv_full;
    uint64_t q_full[2];              // Q and dO of stage s loaded
    uint64_t q_empty[2];             // stage s free (the tile's MMAs are done)
    uint64_t s_full;                 // S^T in TMEM
    uint64_t dp_full;                // dP^T in TMEM
    uint64_t p_ready;                // P8^T in shared memory (both softmax warpgroups)
    uint64_t ds_ready;               // dS8^T in shared memory
    uint64_t dq_full;
    uint64_t dq_free;
    uint64_t dkv_full;
    uint64_t stats_full[2];          // LSE2 / Delta buffer written (count 32)
    uint64_t dstage_full[4];         // dQ_part slice j staged (count 128)
    uint64_t dstage_free;            // the staging buffer has been read by the reductions
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// Shared memory: K, V (one tile each), Q and dO (two stages each), the P8^T
// and dS8^T tiles (128 keys x 128 queries, 128-byte swizzle), the dQ staging
// buffer (D/64 slices of 128 rows x 64 bf16, 128-byte swizzle), LSE2 / Delta
// in two buffers, barriers.
template <int D>
struct Layout {
    static_assert(D == 64 || D == 128, "head dim");
    static constexpr int kRowBytes = D;                                // 8-bit elements
    static constexpr int kSwz = kRowBytes;                             // 64 or 128
    static constexpr uint32_t kSwzCode = (kSwz == 128) ? 2u : 4u;
    static constexpr int kTileBytes = kBlockM * kRowBytes;
    static constexpr int kSbo = 8 * kSwz;
    static constexpr int kSteps = kRowBytes / 32;                      // K = D MMAs: 32 elements each
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kTileBytes;
    static constexpr int kOffQ = kOffV + kTileBytes;                   // 2 stages
    static constexpr int kOffDO = kOffQ + 2 * kTileBytes;              // 2 stages
    static constexpr int kOffPT = kOffDO + 2 * kTileBytes;             // 128 x 128 bytes
    static constexpr int kOffDS = kOffPT + kBlockN * 128;
    static constexpr int kOffStage = kOffDS + kBlockN * 128;           // 128 x D bf16
    static constexpr int kStageBytes = kBlockM * D * 2;
    static constexpr int kOffStats = kOffStage + kStageBytes;
    static constexpr int kOffBar = kOffStats + 2 * 2 * kBlockM * 4;
    static constexpr int kSmemBytes = kOffBar + 256;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(kOffPT % 1024 == 0 && kOffStage % 1024 == 0, "swizzled tiles need 1024-byte alignment");
    static_assert(sizeof(Barriers) <= 256, "barrier block");
    static_assert(D / 64 <= 4 && kStageBytes == (D / 64) * kSliceBytes, "staging: one barrier per 64-column slice");
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
    static_assert(kColDK + D <= 512, "TMEM columns");
};

// kind::f8f6f4 instruction descriptor with separate A / B formats
// (0 = E4M3, 1 = E5M2), fp32 accumulator, and A / B major-ness.
__host__ __device__ constexpr uint32_t idesc_f8(uint32_t a_fmt, uint32_t b_fmt, int M, int N, bool a_mn, bool b_mn)
{
    return (1u << 4) | (a_fmt << 7) | (b_fmt << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kE4M3 = 0, kE5M2 = 1;

// Two floats -> two E5M2 bytes (round to nearest even, saturate to +-57344):
// `lo` in the low byte.
__device__ __forceinline__ uint16_t f32x2_to_e5m2x2(float lo, float hi)
{
    uint16_t h;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(h) : "f"(hi), "f"(lo));
    return h;
}

// Two E5M2 bytes -> f16x2 (exact: E5M2 is f16 with the low 8 bits cleared).
__device__ __forceinline__ uint32_t e5m2x2_to_f16x2(uint16_t v)
{
    uint32_t r;
    asm("cvt.rn.f16x2.e5m2x2 %0, %1;" : "=r"(r) : "h"(v));
    return r;
}


template <int D>
__global__ void __launch_bounds__(kThreads, 1)
sdpa_bwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_dq, const Params p)
{
    using L = Layout<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {
        // the layout relies on the declared alignment; never seen otherwise
        if (threadIdx.x == 0)
            atomicCAS(&g_sdpa_error, 0u, kErrBwd8Wait + 31);
        return;
    }
    uint8_t* smem = smem_raw;
    auto* bars = reinterpret_cast<Barriers*>(smem + L::kOffBar);
    volatile int* abort = &bars->abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // this CTA: key tile kt of KV head hkv of batch b; key tiles ascending
    // over the grid (under the causal mask the longest CTAs start first)
    const int n_bg = p.B * p.Hkv;
    const int kt = blockIdx.x / n_bg;
    const int bg = blockIdx.x % n_bg;
    const int hkv = bg % p.Hkv;
    const int b = bg / p.Hkv;
    const int qt0 = p.causal ? kt : 0;
    const int n_q = p.n_qt > qt0 ? p.n_qt - qt0 : 0;
    const int n_iter = n_q * p.group;            // (head, query tile) pairs, head-major

    const uint32_t sK = smem_u32(smem + L::kOffK);
    const uint32_t sV = smem_u32(smem + L::kOffV);
    const uint32_t sQ = smem_u32(smem + L::kOffQ);
    const uint32_t sDO = smem_u32(smem + L::kOffDO);
    const uint32_t sPT = smem_u32(smem + L::kOffPT);
    const uint32_t sDS = smem_u32(smem + L::kOffDS);
    const uint32_t sStage = smem_u32(smem + L::kOffStage);
    float* stats = reinterpret_cast<float*>(smem + L::kOffStats);      // [2][LSE2 128 | Delta 128]

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars->kv_full), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&bars->q_full[s]), 1);
            mbar_init(smem_u32(&bars->q_empty[s]), 1);
            mbar_init(smem_u32(&bars->stats_full[s]), 32);
        }
        mbar_init(smem_u32(&bars->s_full), 1);
        mbar_init(smem_u32(&bars->dp_full), 1);
        mbar_init(smem_u32(&bars->p_ready), 256);          // both softmax warpgroups
        mbar_init(smem_u32(&bars->ds_ready), 256);
        mbar_init(smem_u32(&bars->dq_full), 1);
        mbar_init(smem_u32(&bars->dq_free), 128);
        mbar_init(smem_u32(&bars->dkv_full), 1);
        for (int j = 0; j < 4; ++j)
            mbar_init(smem_u32(&bars->dstage_full[j]), 128);
        mbar_init(smem_u32(&bars->dstage_free), 1);
        mbar_init(smem_u32(&bars->drain), 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&bars->tmem_base), 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    // programmatic dependent launch: global memory only after the previous
    // kernel in the stream (the Delta pass) has completed
    grid_dependency_wait();
    grid_launch_dependents();
    // (head, query tile) of iteration it: head-major with ascending query
    // tiles; for causal passes with 8 or more query heads per KV head, query
    // tiles from the last down with the heads innermost, so that the CTAs of
    // a KV head work on the same few query tiles at a time (measured on one
    // box: causal MQA S=4096 846 against 785 TFLOP/s; non-causal MQA 958
    // against 1030 and GQA with 4 heads -2 %, which keep the first order)
    const bool heads_inner = p.causal && p.group >= 8;
    auto head_of = [&](int it) { return hkv * p.group + (heads_inner ? it % p.group : it / n_q); };
    auto qtile_of = [&](int it) { return heads_inner ? p.n_qt - 1 - it / p.group : qt0 + it % n_q; };

    if (warp < kSoftmaxWarp0) {
      regs_release<kRegsLow>();
      if (warp == kProducerWarp) {
        // =========================== TMA producer ===========================
        if (lane == 0 && n_iter > 0) {
            tma_prefetch_map(&tm_q);
            tma_prefetch_map(&tm_k);
            tma_prefetch_map(&tm_v);
            tma_prefetch_map(&tm_do);
            mbar_arrive_expect_tx(smem_u32(&bars->kv_full), 2 * L::kTileBytes);
            tma_load_4d(sK, &tm_k, smem_u32(&bars->kv_full), 0, hkv, kt * kBlockN, b);
            tma_load_4d(sV, &tm_v, smem_u32(&bars->kv_full), 0, hkv, kt * kBlockN, b);
            int issued = 0;
            for (int it = 0; it < n_iter; ++it) {
                const int s = it & 1;
                if (it >= 2 &&
                    !wait_bar(smem_u32(&bars->q_empty[s]), ((it >> 1) & 1) ^ 1, abort, kErrBwd8Wait + 1))
                    break;
                const int h = head_of(it), qt = qtile_of(it);
                mbar_arrive_expect_tx(smem_u32(&bars->q_full[s]), 2 * L::kTileBytes);
                tma_load_4d(sQ + s * L::kTileBytes, &tm_q, smem_u32(&bars->q_full[s]), 0, h, qt * kBlockM, b);
                tma_load_4d(sDO + s * L::kTileBytes, &tm_do, smem_u32(&bars->q_full[s]), 0, h, qt * kBlockM, b);
                ++issued;
            }
            {
                // never leave the CTA with copies in flight: the last phase of
                // every slot (complete already in a normal run; after an
                // abort, the copies still landing)
                drain_wait(smem_u32(&bars->kv_full), 0);
                for (int it = (issued > 2 ? issued - 2 : 0); it < issued; ++it)
                    drain_wait(smem_u32(&bars->q_full[it & 1]), (it >> 1) & 1);
            }
        }
      } else if (warp == kMmaWarp) {
        // ============================ MMA issuer ============================
        if (lane == 0 && n_iter > 0) {
            constexpr uint32_t id_s = idesc_f8(kE4M3, kE4M3, kBlockM, kBlockN, false, false);   // K Q^T
            constexpr uint32_t id_dp = idesc_f8(kE4M3, kE5M2, kBlockM, kBlockN, false, false);  // V dO^T
            constexpr uint32_t id_dv = idesc_f8(kE4M3, kE5M2, kBlockM, D, false, true);         // P8^T dO
            constexpr uint32_t id_dk = idesc_f8(kE5M2, kE4M3, kBlockM, D, false, true);         // dS8^T Q
            constexpr uint32_t id_dq = idesc_f8(kE5M2, kE4M3, kBlockM, D, true, true);          // dS8 K
            // descriptors as (hi, lo) halves: the D-byte operand tiles and
            // the 128-byte P8^T / dS8^T tiles (LBO unused: one swizzle atom wide)
            const uint32_t hi = (uint32_t)(smem_desc(0, 16, L::kSbo, L::kSwzCode) >> 32);
            const uint32_t hi_t = (uint32_t)(smem_desc(0, 16, 1024, 2u) >> 32);
            const uint32_t lbo = 1u << 16;
            const uint32_t k_lo = (sK >> 4) | lbo, v_lo = (sV >> 4) | lbo;
            const uint32_t pt_lo = (sPT >> 4) | lbo, ds_lo = (sDS >> 4) | lbo;
            const uint32_t s_t = tmem + L::kColS, dp_t = tmem + L::kColDP;
            const uint32_t dv_t = tmem + L::kColDV, dk_t = tmem + L::kColDK;
            // S^T = K Q^T (keys x queries, K = D) of tile `it` into cols 0..127
            auto issue_s = [&](int it) -> bool {
                const int s = it & 1;
                if (!wait_bar(smem_u32(&bars->q_full[s]), (it >> 1) & 1, abort, kErrBwd8Wait + 3))
                    return false;
                tc_fence_after_sync();
                const uint32_t q_lo = ((sQ + s * L::kTileBytes) >> 4) | lbo;
#pragma unroll
                for (int kk = 0; kk < L::kSteps; ++kk)
                    mma_f8_ss(s_t, desc_join(hi, k_lo + 2 * kk), desc_join(hi, q_lo + 2 * kk), id_s, kk > 0);
                mma_commit(smem_u32(&bars->s_full));
                return true;
            };
            bool ok = wait_bar(smem_u32(&bars->kv_full), 0, abort, kErrBwd8Wait + 2);
            if (ok)
                ok = issue_s(0);
            for (int it = 0; ok && it < n_iter; ++it) {
                const int s = it & 1;
                bool s_next = it + 1 >= n_iter;             // the next tile's S^T issued
                const uint32_t q_lo = ((sQ + s * L::kTileBytes) >> 4) | lbo;
                const uint32_t do_lo = ((sDO + s * L::kTileBytes) >> 4) | lbo;
                // dP^T = V dO^T into cols 128..255, once the dQ warps have read the
                // last tile's dQ_part out of them
                if (it > 0 && !(ok = wait_bar(smem_u32(&bars->dq_free), (it - 1) & 1, abort, kErrBwd8Wait + 4)))
                    break;
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < L::kSteps; ++kk)
                    mma_f8_ss(dp_t, desc_join(hi, v_lo + 2 * kk), desc_join(hi, do_lo + 2 * kk), id_dp, kk > 0);
                mma_commit(smem_u32(&bars->dp_full));
                // dV += P8^T dO: 32 queries per step, P8^T K-major (32 bytes
                // of its rows), dO MN-major (32 of its rows)
                if (!(ok = wait_bar(smem_u32(&bars->p_ready), it & 1, abort, kErrBwd8Wait + 5)))
                    break;
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < kBlockM / 32; ++kk) {
                    const uint32_t off = (uint32_t)((kk * 32 * L::kRowBytes) >> 4);
                    mma_f8_ss(dv_t, desc_join(hi_t, pt_lo + 2 * kk), desc_join(hi, do_lo + off), id_dv,
                              (it > 0 || kk > 0) ? 1u : 0u);
                }
                // the next tile's S^T after this dV MMA (the last reader of the
                // P8^T tile the next softmax writes) if its Q has landed
                if (!s_next && mbar_test_wait(smem_u32(&bars->q_full[(it + 1) & 1]), ((it + 1) >> 1) & 1)) {
                    if (!(ok = issue_s(it + 1)))
                        break;
                    s_next = true;
                }
                // dQ_part = dS8 K first, into cols 128..128+D-1 (free once the
                // softmax has read dP^T), so that its read-out frees them for
                // the next dP^T: A = the dS8^T tile read MN-major (32 key rows
                // per step), K MN-major (32 key rows per step)
                if (!(ok = wait_bar(smem_u32(&bars->ds_ready), it & 1, abort, kErrBwd8Wait + 6)))
                    break;
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < kBlockN / 32; ++kk) {
                    const uint32_t off_a = (uint32_t)((kk * 32 * 128) >> 4);
                    const uint32_t off_b = (uint32_t)((kk * 32 * L::kRowBytes) >> 4);
                    mma_f8_ss(dp_t, desc_join(hi_t, ds_lo + off_a), desc_join(hi, k_lo + off_b), id_dq, kk > 0);
                }
                mma_commit(smem_u32(&bars->dq_full));
                // dK += dS8^T Q: dS8^T K-major, Q MN-major
#pragma unroll
                for (int kk = 0; kk < kBlockM / 32; ++kk) {
                    const uint32_t off = (uint32_t)((kk * 32 * L::kRowBytes) >> 4);
                    mma_f8_ss(dk_t, desc_join(hi_t, ds_lo + 2 * kk), desc_join(hi, q_lo + off), id_dk,
                              (it > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(smem_u32(&bars->q_empty[s]));     // the dK MMA was Q's last reader
                if (!s_next && !(ok = issue_s(it + 1)))
                    break;
            }
            mma_commit(smem_u32(&bars->dkv_full));
            mma_commit(smem_u32(&bars->drain));
            drain_wait(smem_u32(&bars->drain), 0);
        }
      } else if (warp == kReduceWarp) {
        // ==================== dQ_part into the bf16 accumulator ==============
        // The reductions run at a fixed number of bytes per cycle on an SM
        // (measured: ~24 B/cycle into L2, bf16 and fp32 alike), so a bf16
        // accumulator halves the time they take; its rounding (~1 % relative
        // over the causal pass's key tiles) is far below the E5M2 rounding of
        // dS that bounds this pass's dQ.
        if (lane == 0 && n_iter > 0) {
            tma_prefetch_map(&tm_dq);
            for (int it = 0; it < n_iter; ++it) {
                const int h = head_of(it), qt = qtile_of(it);
                bool staged = true;
                for (int j = 0; j < D / 64; ++j) {
                    if (!(staged = wait_bar(smem_u32(&bars->dstage_full[j]), it & 1, abort, kErrBwd8Wait + 7)))
                        break;
                    tma_reduce_add_4d(&tm_dq, sStage + (uint32_t)(j * kSliceBytes), 64 * j, h, qt * kBlockM, b);
                }
                bulk_commit_group();
                if (!staged)
                    break;
                bulk_wait_group_read0();                    // the staging buffer may be rewritten
                mbar_arrive(smem_u32(&bars->dstage_free));
            }
            bulk_wait_group0();                             // the reductions have landed
        }
      } else if (warp == kStatsWarp) {
        // ====================== LSE2 / Delta of each tile =====================
        // As in the 16-bit kernel: four query rows per lane, buffer it & 1,
        // written once p_ready of tile it - 1 shows its last readers done.
        for (int it = 0; it < n_iter; ++it) {
            if (it > 0 &&
                !__all_sync(0xffffffffu, wait_bar(smem_u32(&bars->p_ready), (it - 1) & 1, abort, kErrBwd8Wait + 8)))
                break;
            const int qr0 = qtile_of(it) * kBlockM + 4 * lane;
            const int64_t row = ((int64_t)b * p.Hq + head_of(it)) * p.Sq;
            float l2[4], dl[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const bool v = qr0 + e < p.Sq;
                l2[e] = v ? p.lse[row + qr0 + e] * kLog2e : INFINITY;
                dl[e] = v ? p.delta[row + qr0 + e] : 0.f;
            }
            float4* buf = reinterpret_cast<float4*>(stats + (it & 1) * 2 * kBlockM);
            buf[lane] = make_float4(l2[0], l2[1], l2[2], l2[3]);
            buf[kBlockM / 4 + lane] = make_float4(dl[0], dl[1], dl[2], dl[3]);
            mbar_arrive(smem_u32(&bars->stats_full[it & 1]));
        }
      }
    } else if (warp < kDqWarp0) {
        regs_acquire<kRegsSoftmax>();
        // ============ P8^T and dS8^T, one thread per key row ==============
        const int sw = (warp - kSoftmaxWarp0) >> 2;         // query half of this warpgroup
        const int quarter = warp & 3;
        const int kr = quarter * 32 + lane;                 // key row of the tile (= TMEM lane)
        const int key = kt * kBlockN + kr;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const uint32_t s_t = tmem + lane_addr + L::kColS;
        const uint32_t dp_t = tmem + lane_addr + L::kColDP;
        const bool key_ok = key < p.Skv;
        // this key's rows of the P8^T / dS8^T tiles (128 queries, 128-byte swizzle)
        const uint32_t pt_row = sPT + (uint32_t)(kr * 128), ds_row = sDS + (uint32_t)(kr * 128);
        float amax = 0.f;                                   // max |dS P-scaled| seen by this thread
        bool ok = true;
        for (int it = 0; ok && it < n_iter; ++it) {
            ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->s_full), it & 1, abort, kErrBwd8Wait + 9));
            if (ok)
                ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->stats_full[it & 1]), (it >> 1) & 1, abort,
                                                      kErrBwd8Wait + 10));
            if (!ok)
                break;
            tc_fence_after_sync();
            const float4* l2v = reinterpret_cast<const float4*>(stats + (it & 1) * 2 * kBlockM);
            const float4* dlv = l2v + kBlockM / 4;
            // top-left causal: this key is visible to query q iff key <= q;
            // keys past Skv are visible to none
            const int first_q = !key_ok ? (1 << 30) : (p.causal ? key - qtile_of(it) * kBlockM : -1);
            // phase 1, from S^T alone: P (kept in fp32 for dS) and P8 = e4m3(448 P)
            // into bytes 64 sw .. 64 sw + 63 of the row
            float pf[2][32];
#pragma unroll
            for (int chh = 0; chh < 2; ++chh) {             // 32 queries per chunk, two per warpgroup
                const int ch = 2 * sw + chh;
                uint32_t sv[32];
                tmem_ld32_wait(s_t + 32 * ch, sv);
                uint32_t pk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 l4 = l2v[8 * ch + i];
                    const float lq[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int q = 32 * ch + 4 * i + e;
                        pf[chh][4 * i + e] =
                            q >= first_q ? ex2_approx(__uint_as_float(sv[4 * i + e]) * p.c_s - lq[e]) : 0.f;
                    }
                    pk[i] = (uint32_t)f32x2_to_e4m3x2(pf[chh][4 * i] * kPScale, pf[chh][4 * i + 1] * kPScale) |
                            ((uint32_t)f32x2_to_e4m3x2(pf[chh][4 * i + 2] * kPScale, pf[chh][4 * i + 3] * kPScale)
                             << 16);
                }
                // queries 32 ch .. 32 ch + 31 are 16-byte units 2 ch, 2 ch + 1
#pragma unroll
                for (int uu = 0; uu < 2; ++uu) {
                    const int u = 2 * ch + uu;
                    st_shared_v4(pt_row + (uint32_t)((u ^ (kr & 7)) << 4), pk[4 * uu], pk[4 * uu + 1],
                                 pk[4 * uu + 2], pk[4 * uu + 3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(smem_u32(&bars->p_ready));          // dV += P8^T dO can start
            // phase 2, once dP^T is there: dS = P (dv dP - Delta) in units of
            // ddo, and dS8 = e5m2(ddo scale_ds dS) into the dS8^T row
            ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->dp_full), it & 1, abort, kErrBwd8Wait + 11));
            if (!ok)
                break;
            tc_fence_after_sync();
#pragma unroll
            for (int chh = 0; chh < 2; ++chh) {
                const int ch = 2 * sw + chh;
                uint32_t dv[32];
                tmem_ld32_wait(dp_t + 32 * ch, dv);
                uint32_t dk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 d4 = dlv[8 * ch + i];
                    const float dq[4] = {d4.x, d4.y, d4.z, d4.w};
                    float ds[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        ds[e] = pf[chh][4 * i + e] * (__uint_as_float(dv[4 * i + e]) * p.dv - dq[e]);
                        amax = fmaxf(amax, fabsf(ds[e]));
                    }
                    dk[i] = (uint32_t)f32x2_to_e5m2x2(ds[0] * p.m_ds, ds[1] * p.m_ds) |
                            ((uint32_t)f32x2_to_e5m2x2(ds[2] * p.m_ds, ds[3] * p.m_ds) << 16);
                }
#pragma unroll
                for (int uu = 0; uu < 2; ++uu) {
                    const int u = 2 * ch + uu;
                    st_shared_v4(ds_row + (uint32_t)((u ^ (kr & 7)) << 4), dk[4 * uu], dk[4 * uu + 1],
                                 dk[4 * uu + 2], dk[4 * uu + 3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(smem_u32(&bars->ds_ready));
        }
        // amax |dS| of this call (non-negative floats order as their bits)
#pragma unroll
        for (int s = 16; s > 0; s >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, s));
        if (lane == 0)
            atomicMax(p.amax_ds, __float_as_uint(amax * p.ddo));
        // ---- dK, dV of this key: the accumulators times their output factor ----
        if (ok && n_iter > 0) {
            ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->dkv_full), 0, abort, kErrBwd8Wait + 12));
            tc_fence_after_sync();
        }
        if (ok) {
            const int64_t row_off = (((int64_t)b * p.Skv + key) * p.Hkv + hkv) * D;
            const int which = sw;                           // first warpgroup dV, second dK
            uint16_t* dst = reinterpret_cast<uint16_t*>(which ? p.dK : p.dV) + row_off;
            const uint32_t col = which ? L::kColDK : L::kColDV;
            const float f = which ? p.out_dk : p.out_dv;
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t r[32];
                if (n_iter > 0) {
                    tmem_ld32_wait(tmem + lane_addr + col + 32 * cc, r);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        r[i] = 0u;                          // no query sees this key
                }
                if (key_ok) {
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        reinterpret_cast<uint4*>(dst + 32 * cc)[v] = make_uint4(
                            pack2<true>(f * __uint_as_float(r[8 * v]), f * __uint_as_float(r[8 * v + 1])),
                            pack2<true>(f * __uint_as_float(r[8 * v + 2]), f * __uint_as_float(r[8 * v + 3])),
                            pack2<true>(f * __uint_as_float(r[8 * v + 4]), f * __uint_as_float(r[8 * v + 5])),
                            pack2<true>(f * __uint_as_float(r[8 * v + 6]), f * __uint_as_float(r[8 * v + 7])));
                }
            }
        }
    } else {
        regs_acquire<kRegsDq>();
        // ============ dQ_part out of TMEM into the staging buffer =============
        const int quarter = warp & 3;
        const int qr = quarter * 32 + lane;                 // query row of the tile (= TMEM lane)
        const uint32_t src = tmem + ((uint32_t)(quarter * 32) << 16) + L::kColDP;   // dQ_part
        bool ok = true;
        for (int it = 0; ok && it < n_iter; ++it) {
            ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->dq_full), it & 1, abort, kErrBwd8Wait + 13));
            if (!ok)
                break;
            tc_fence_after_sync();
            uint32_t r[D];
#pragma unroll
            for (int c = 0; c < D / 32; ++c)
                tmem_ld32_wait(src + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * c]));
            tc_fence_before_sync();
            mbar_arrive(smem_u32(&bars->dq_free));
            // the buffer is free once the last tile's reductions have read it
            if (it > 0)
                ok = __all_sync(0xffffffffu,
                                wait_bar(smem_u32(&bars->dstage_free), (it - 1) & 1, abort, kErrBwd8Wait + 14));
            if (!ok)
                break;
            // bf16, 64-column slices of 128 rows x 128 bytes, 128-byte swizzle
#pragma unroll
            for (int j = 0; j < D / 64; ++j) {
                const uint32_t row = sStage + (uint32_t)(j * kSliceBytes + qr * 128);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int e = 64 * j + 8 * u;
                    st_shared_v4(row + (uint32_t)((u ^ (qr & 7)) << 4),
                                 pack2<true>(__uint_as_float(r[e]), __uint_as_float(r[e + 1])),
                                 pack2<true>(__uint_as_float(r[e + 2]), __uint_as_float(r[e + 3])),
                                 pack2<true>(__uint_as_float(r[e + 4]), __uint_as_float(r[e + 5])),
                                 pack2<true>(__uint_as_float(r[e + 6]), __uint_as_float(r[e + 7])));
                }
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&bars->dstage_full[j]));   // the reducer may start on it
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

// Delta8_i = sum_d dO8_id O_id (fp32): dO as E5M2 codes (one byte each), O
// 16-bit, both [B][Sq][Hq][D]; written to the [B][Hq][Sq] layout.  One
// group of D / 16 lanes per row, 16 codes (16 bytes) a lane, two rows a
// group.  The same pass zeroes the row's D bf16 of the dQ accumulator
// ([B][Sq][Hq][D]) and the amax word: one launch instead of two memsets and
// this kernel.
template <int D, bool kBF16>
__global__ void __launch_bounds__(256) bwd8_delta_kernel(const void* O, const void* dO8, float* delta,
                                                         uint16_t* dq_acc, unsigned int* amax, int B, int Hq, int Sq)
{
    grid_dependency_wait();                       // launched with programmatic serialization
    grid_launch_dependents();
    constexpr int kLanes = D / 16;
    constexpr int kGroups = 256 / kLanes;
    const int64_t rows = (int64_t)B * Sq * Hq;
    const int c = threadIdx.x % kLanes;
    if (blockIdx.x == 0 && threadIdx.x == 0)
        *amax = 0u;                                     // the main kernel's atomic max starts from 0
    int64_t row[2];
    uint4 g[2], o0[2], o1[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        row[k] = (int64_t)blockIdx.x * (2 * kGroups) + k * kGroups + threadIdx.x / kLanes;
        if (row[k] < rows) {
            g[k] = reinterpret_cast<const uint4*>(dO8)[row[k] * kLanes + c];
            const uint4* o = reinterpret_cast<const uint4*>(O) + (row[k] * kLanes + c) * 2;
            o0[k] = o[0];
            o1[k] = o[1];
        }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        float acc = 0.f;
        if (row[k] < rows) {
            uint4* z = reinterpret_cast<uint4*>(dq_acc + row[k] * D + 16 * c);
            z[0] = make_uint4(0u, 0u, 0u, 0u);
            z[1] = make_uint4(0u, 0u, 0u, 0u);
            const uint32_t gv[4] = {g[k].x, g[k].y, g[k].z, g[k].w};
            const uint32_t ov[8] = {o0[k].x, o0[k].y, o0[k].z, o0[k].w, o1[k].x, o1[k].y, o1[k].z, o1[k].w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const uint32_t g2 = e5m2x2_to_f16x2((uint16_t)(gv[e / 2] >> (16 * (e & 1))));
                const float2 gf = __half22float2(*reinterpret_cast<const __half2*>(&g2));
                float2 of;
                if constexpr (kBF16)
                    of = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ov[e]));
                else
                    of = __half22float2(*reinterpret_cast<const __half2*>(&ov[e]));
                acc = fmaf(gf.x, of.x, acc);
                acc = fmaf(gf.y, of.y, acc);
            }
        }
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

// dQ (bf16, [B][Sq][Hq][D]) = factor * the bf16 accumulator, 8 elements a thread.
__global__ void __launch_bounds__(256) bwd8_dq_convert_kernel(const uint16_t* acc, void* dQ, int64_t n, float factor)
{
    grid_dependency_wait();                       // launched with programmatic serialization
    grid_launch_dependents();
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
    if (i >= n)
        return;
    const uint4 v = *reinterpret_cast<const uint4*>(acc + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xffff0000u);   // bf16 -> fp32, exact
        o[k] = pack2<true>(factor * lo, factor * hi);
    }
    *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(dQ) + i) = make_uint4(o[0], o[1], o[2], o[3]);
}

}  // namespace bwd8
}  // namespace sdpa
