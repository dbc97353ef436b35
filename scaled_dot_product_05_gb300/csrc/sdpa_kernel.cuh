// sdpa_kernel.cuh -- fused attention forward pass for sm_103a.
//
// Computes O = softmax(Q K^T * scale [+ causal mask]) V, the definition in the
// codelab "Attention on GPU (cuDNN and TransformerEngine)", section 1 ("How
// attention works"), in one pass over the keys with a running max and sum
// (online softmax), so the Sq x Skv score matrix never leaves the chip -- the
// tiling that section 8 ("Run benchmarks", sequence sweep) credits fused
// kernels with.
//
// One CTA computes one work unit: 128 query rows of one (batch, query head).
// Warp roles:
//   warp 0      TMA producer: the Q tile once, then K_j and V_j tiles into
//               two- or three-stage shared-memory rings.
//   warp 1      tcgen05 issuer: S_j = Q K_j^T into one of two TMEM score
//               buffers, and O += P_j V_j with P_j read from TMEM.
//   warps 2..5  softmax warpgroup: one thread per query row reads its S row
//               from TMEM, applies the causal / tail mask, updates the
//               running max m and sum l, writes P = exp2(S*c - m) as 16-bit
//               values back over its S row, rescales O in TMEM when m moved,
//               and finally writes O / l to global memory.
//
// Layout: Q, O are [B][Sq][Hq][D] and K, V are [B][Skv][Hkv][D] (section 3,
// "Create Q, K and V test arrays": (B, T, N, H)).  Query head hq reads KV head
// hq / (Hq / Hkv) (section 9, "Compare MHA, GQA and MQA"); nothing is
// replicated.  Causal masking keeps the lower triangle (section 7, "Add causal
// masking"): row i sees keys 0..i; key tiles wholly above the diagonal are
// skipped and only the diagonal tile is masked element-wise.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace sdpa {

constexpr int kBlockM = 128;         // query rows per work unit (= TMEM lanes)
constexpr int kBlockN = 128;         // keys per K/V tile
constexpr int kThreads = 192;        // 6 warps
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s per barrier wait

// Device error word: 0 = no error; otherwise the first failure recorded by any
// CTA (see the codes below).  Read and cleared by the host through the C-ABI.
__device__ unsigned int g_sdpa_error = 0;

enum : unsigned int {
    kErrWaitLoad = 0x100,            // + barrier id: producer wait timed out
    kErrWaitMma = 0x200,             // + barrier id: MMA issuer wait timed out
    kErrWaitSoftmax = 0x300,         // + barrier id: softmax wait timed out
};

struct Params {
    void* O;
    int B, Hq, Hkv, Sq, Skv;
    int group;                       // Hq / Hkv
    int n_qtiles;                    // ceil(Sq / 128)
    int n_ktiles;                    // ceil(Skv / 128)
    int causal;
    float scale_log2;                // scale * log2(e): scores enter exp2
};

template <int D>
struct Layout {
    static constexpr int kChunks = D / 64;                   // 128-byte swizzle column blocks
    static constexpr int kChunkBytes = kBlockM * 128;         // 128 rows x 128 B
    static constexpr int kTileBytes = kBlockM * D * 2;        // one Q, K or V tile
    static constexpr int kStages = (D == 128) ? 2 : 3;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kTileBytes;
    static constexpr int kOffV = kOffK + kStages * kTileBytes;
    static constexpr int kOffBar = kOffV + kStages * kTileBytes;
    static constexpr int kBarBytes = 512;
    // Request at least ~116 KB so that only one CTA (which takes all 512 TMEM
    // columns) is resident per SM.
    static constexpr int kUsed = kOffBar + kBarBytes;
    static constexpr int kSmemBytes = (kUsed > 118 * 1024 ? kUsed : 118 * 1024) + 1024;
    // TMEM columns
    static constexpr uint32_t kTmemS0 = 0;
    static constexpr uint32_t kTmemS1 = 128;
    static constexpr uint32_t kTmemO = 256;
    static constexpr uint32_t kTmemCols = 512;
};

template <int kStages>
struct Barriers {
    uint64_t q_full;
    uint64_t k_full[kStages];
    uint64_t k_empty[kStages];
    uint64_t v_full[kStages];
    uint64_t v_empty[kStages];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_done;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// Bounded wait: gives up after kWaitLimitNs, records `code` in the device
// error word, and raises the CTA's abort flag so that every later wait in the
// CTA returns at once.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort, unsigned int code)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*abort)
            return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            atomicCAS(&g_sdpa_error, 0u, code);
            return false;
        }
    }
}

template <bool kBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    if constexpr (kBF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

template <int D, bool kBF16>
__global__ void __launch_bounds__(kThreads, 1)
sdpa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const Params p)
{
    using L = Layout<D>;
    constexpr int NS = L::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    auto* bars = reinterpret_cast<Barriers<NS>*>(smem + L::kOffBar);
    volatile int* abort = &bars->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // ---- work unit: heaviest causal tiles (largest q-tile index) first ------
    const int bh_count = p.B * p.Hq;
    int qt = blockIdx.x / bh_count;
    if (p.causal)
        qt = p.n_qtiles - 1 - qt;
    const int bh = blockIdx.x % bh_count;
    const int b = bh / p.Hq;
    const int hq = bh % p.Hq;
    const int hkv = hq / p.group;
    const int n_kv = p.causal ? min(p.n_ktiles, qt + 1) : p.n_ktiles;

    const uint32_t sQ = smem_u32(smem + L::kOffQ);
    const uint32_t sK = smem_u32(smem + L::kOffK);
    const uint32_t sV = smem_u32(smem + L::kOffV);

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars->q_full), 1);
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&bars->k_full[s]), 1);
            mbar_init(smem_u32(&bars->k_empty[s]), 1);
            mbar_init(smem_u32(&bars->v_full[s]), 1);
            mbar_init(smem_u32(&bars->v_empty[s]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&bars->s_full[i]), 1);
            mbar_init(smem_u32(&bars->p_full[i]), 128);
        }
        mbar_init(smem_u32(&bars->o_done), 1);
        mbar_init(smem_u32(&bars->drain), 1);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&tm_q);
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_v);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_base), L::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // =========================== TMA producer ===========================
        if (lane == 0) {
            const int q0 = qt * kBlockM;
            mbar_arrive_expect_tx(smem_u32(&bars->q_full), L::kTileBytes);
            for (int c = 0; c < L::kChunks; ++c)
                tma_load_4d(sQ + c * L::kChunkBytes, &tm_q, smem_u32(&bars->q_full), c * 64, hq, q0, b);
            int nk = 0, nv = 0;                              // K / V tiles issued
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % NS;
                const uint32_t par = ((j / NS) & 1) ^ 1;     // phase of the release of tile j - NS
                if (j >= NS && !wait_bar(smem_u32(&bars->k_empty[s]), par, abort, kErrWaitLoad + 1))
                    break;
                mbar_arrive_expect_tx(smem_u32(&bars->k_full[s]), L::kTileBytes);
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_4d(sK + s * L::kTileBytes + c * L::kChunkBytes, &tm_k, smem_u32(&bars->k_full[s]),
                                c * 64, hkv, j * kBlockN, b);
                nk = j + 1;
                if (j >= NS && !wait_bar(smem_u32(&bars->v_empty[s]), par, abort, kErrWaitLoad + 2))
                    break;
                mbar_arrive_expect_tx(smem_u32(&bars->v_full[s]), L::kTileBytes);
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_4d(sV + s * L::kTileBytes + c * L::kChunkBytes, &tm_v, smem_u32(&bars->v_full[s]),
                                c * 64, hkv, j * kBlockN, b);
                nv = j + 1;
            }
            // Never leave the CTA with copies in flight: after an abort, wait
            // (bounded) for the last copy issued into every stage.
            if (*abort) {
                auto drain = [&](uint32_t bar, uint32_t parity) {
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(bar, parity) && global_timer_ns() - t0 < kWaitLimitNs) {
                    }
                };
                drain(smem_u32(&bars->q_full), 0);
                for (int j = (nk > NS ? nk - NS : 0); j < nk; ++j)
                    drain(smem_u32(&bars->k_full[j % NS]), (j / NS) & 1);
                for (int j = (nv > NS ? nv - NS : 0); j < nv; ++j)
                    drain(smem_u32(&bars->v_full[j % NS]), (j / NS) & 1);
            }
        }
    } else if (warp == 1) {
        // ============================ MMA issuer ============================
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_f16(kBF16, kBlockM, kBlockN, false);
            constexpr uint32_t idesc_o = idesc_f16(kBF16, kBlockM, D, true);
            bool ok = wait_bar(smem_u32(&bars->q_full), 0, abort, kErrWaitMma + 0);
            tc_fence_after_sync();
            // S_j = Q K_j^T into score buffer j & 1.  Q and K tiles are K-major,
            // 128-byte swizzled: 16-element K steps advance 32 bytes inside a
            // 64-column block, blocks are kChunkBytes apart, 8-row groups 1024 B.
            auto issue_s = [&](int j) -> bool {
                const int s = j % NS;
                if (!wait_bar(smem_u32(&bars->k_full[s]), (j / NS) & 1, abort, kErrWaitMma + 1))
                    return false;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem + ((j & 1) ? L::kTmemS1 : L::kTmemS0);
                const uint32_t kbase = sK + s * L::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
                    mma_f16_ss(d_tmem, smem_desc_sw128(sQ + off, 16, 1024), smem_desc_sw128(kbase + off, 16, 1024),
                               idesc_s, kk > 0);
                }
                mma_commit(smem_u32(&bars->s_full[j & 1]));
                mma_commit(smem_u32(&bars->k_empty[s]));
                return true;
            };
            if (ok && n_kv > 0)
                ok = issue_s(0);
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j + 1 < n_kv && !issue_s(j + 1))
                    break;
                const int buf = j & 1;
                if (!wait_bar(smem_u32(&bars->p_full[buf]), (j >> 1) & 1, abort, kErrWaitMma + 2))
                    break;
                tc_fence_after_sync();
                const int s = j % NS;
                if (!wait_bar(smem_u32(&bars->v_full[s]), (j / NS) & 1, abort, kErrWaitMma + 3))
                    break;
                tc_fence_after_sync();
                // O += P_j V_j.  P: 128 x 128 16-bit in TMEM (8 columns per
                // 16 keys).  V tile is MN-major (D contiguous), 128-byte
                // swizzled: 16 keys = 2048 B; the next 64 columns of D are one
                // chunk (kChunkBytes) further.
                const uint32_t p_tmem = tmem + (buf ? L::kTmemS1 : L::kTmemS0);
                const uint32_t vbase = sV + s * L::kTileBytes;
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk) {
                    mma_f16_ts(tmem + L::kTmemO, p_tmem + kk * 8,
                               smem_desc_sw128(vbase + kk * 2048, L::kChunkBytes, 1024), idesc_o,
                               (j > 0 || kk > 0) ? 1u : 0u);
                }
                mma_commit(smem_u32(&bars->v_empty[s]));
                mma_commit(smem_u32(&bars->o_done));
            }
            // Every MMA this thread issued completes before TMEM is released.
            mma_commit(smem_u32(&bars->drain));
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(smem_u32(&bars->drain), 0) && global_timer_ns() - t0 < kWaitLimitNs) {
            }
        }
    } else {
        // ========================= softmax warpgroup ========================
        const int quarter = warp & 3;                      // TMEM lanes 32*quarter ..
        const int row = quarter * 32 + lane;
        const int q_idx = qt * kBlockM + row;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const float c = p.scale_log2;
        int limit = p.Skv - 1;                             // last visible key of this row
        if (p.causal && q_idx < limit)
            limit = q_idx;
        float m = -INFINITY;                               // running max of S*c
        float l = 0.f;                                     // running sum of exp2(S*c - m)
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const int buf = j & 1;
            const uint32_t s_tmem = tmem + lane_addr + (buf ? L::kTmemS1 : L::kTmemS0);
            ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->s_full[buf]), (j >> 1) & 1, abort,
                                                  kErrWaitSoftmax + 1));
            if (!ok)
                break;
            tc_fence_after_sync();
            uint32_t r[128];
            tmem_ld128_wait(s_tmem, s_tmem + 32, s_tmem + 64, s_tmem + 96, r);
            float sv[128];
#pragma unroll
            for (int i = 0; i < 128; ++i)
                sv[i] = __uint_as_float(r[i]);
            const int k0 = j * kBlockN;
            if (k0 + kBlockN - 1 > limit) {
#pragma unroll
                for (int i = 0; i < 128; ++i)
                    if (k0 + i > limit)
                        sv[i] = -INFINITY;
            }
            float mt = sv[0];
#pragma unroll
            for (int i = 1; i < 128; ++i)
                mt = fmaxf(mt, sv[i]);
            const float m_new = fmaxf(m, mt * c);
            const float alpha = ex2_approx(m - m_new);     // 0 on the first tile
            float sum = 0.f;
            uint32_t pk[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const float p0 = ex2_approx(fmaf(sv[2 * i], c, -m_new));
                const float p1 = ex2_approx(fmaf(sv[2 * i + 1], c, -m_new));
                sum += p0 + p1;
                pk[i] = pack2<kBF16>(p0, p1);
            }
            l = l * alpha + sum;
            m = m_new;
            tmem_st32(s_tmem, *reinterpret_cast<const uint32_t(*)[32]>(&pk[0]));
            tmem_st32(s_tmem + 32, *reinterpret_cast<const uint32_t(*)[32]>(&pk[32]));
            // Rescale O by alpha once P_{j-1} V_{j-1} has landed (any row of
            // the warp that moved its max makes the warp do it).
            if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
                ok = __all_sync(0xffffffffu,
                                wait_bar(smem_u32(&bars->o_done), (j - 1) & 1, abort, kErrWaitSoftmax + 2));
                if (!ok)
                    break;
                tc_fence_after_sync();
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t o[32];
                    const uint32_t o_tmem = tmem + lane_addr + L::kTmemO + cc * 32;
                    tmem_ld32_wait(o_tmem, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                    tmem_st32(o_tmem, o);
                }
            }
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(smem_u32(&bars->p_full[buf]));
        }
        // ---- epilogue: O / l -> 16-bit -> global ---------------------------
        if (ok) {
            ok = __all_sync(0xffffffffu,
                            wait_bar(smem_u32(&bars->o_done), (n_kv - 1) & 1, abort, kErrWaitSoftmax + 3));
        }
        if (ok) {
            tc_fence_after_sync();
            const float inv_l = 1.f / l;
            uint8_t* out = reinterpret_cast<uint8_t*>(p.O) +
                           (((int64_t)b * p.Sq + q_idx) * p.Hq + hq) * (int64_t)(D * 2);
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t o[32];
                tmem_ld32_wait(tmem + lane_addr + L::kTmemO + cc * 32, o);
                uint32_t h[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    h[i] = pack2<kBF16>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
                if (q_idx < p.Sq) {
                    uint4* dst = reinterpret_cast<uint4*>(out + cc * 64);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(h[4 * v], h[4 * v + 1], h[4 * v + 2], h[4 * v + 3]);
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

}  // namespace sdpa
