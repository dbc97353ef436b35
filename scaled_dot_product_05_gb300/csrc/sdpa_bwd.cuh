// sdpa_bwd.cuh -- backward pass of the attention forward pass, for sm_103a.
//
// For O = softmax(S) V with S = scale Q K^T (the definition in section 1,
// "How attention works", of the codelab "Attention on GPU (cuDNN and
// TransformerEngine)") and an upstream gradient dO, the chain rule gives
//     P = exp(S - LSE)                     (the forward's row log-sum-exp)
//     dV = P^T dO,   dP = dO V^T,   Delta_i = sum_j P_ij dP_ij = dO_i . O_i
//     dS = P * (dP - Delta),   dQ = scale dS K,   dK = scale dS^T Q.
// The codelab names the backward pass as what training needs (section 10,
// FP8: "E5M2 for the backward pass"); this is its bf16 / fp16 form.
//
// One CTA per (batch, KV head, key tile of 128 keys) owns dK and dV of its
// keys and loops over the query tiles (causal: those on or below its keys)
// of every query head of the group, accumulating in TMEM; key tiles vary
// slowest over the grid, so the longest CTAs start first:
//   warp 0       TMA producer: K, V once; Q and dO tiles into a 2-stage ring,
//                  each with its own full / empty barriers
//   warp 1       tcgen05 issue, per query tile: S^T = K Q^T (cols 0..127;
//                  at D = 64 alternately cols 384..511), dP^T = V dO^T
//                  (cols 128..255); dV += P^T dO once P^T is packed (P^T read
//                  from TMEM); once dS is in shared memory, dQ_part = dS K
//                  (dS an MN-major A operand) into cols 128..128+D-1 first,
//                  so that its read-out frees them for the next dP^T, then
//                  dK += dS^T Q (the same tile as a K-major A operand).  The
//                  next tile's S^T goes in as early as its columns and its Q
//                  allow
//   warp 2       dQ reducer: adds the staged dQ_part of a query tile into
//                  the fp32 dQ accumulator in HBM (TMA bulk reductions), then
//                  hands the tile's Q, then dO, back to the producer
//   warp 3       statistics: LSE2 = LSE log2(e) and Delta of the next tile
//                  into a double-buffered shared array
//   warps 4..11  two warpgroups, one thread per key row each, the first for
//                  queries 0..63 of the tile, the second for 64..127: first
//                  P^T = exp2(S^T c - LSE2) (from S^T alone), packed as
//                  16-bit values over S^T in TMEM, then dS^T = scale P^T
//                  (dP^T - Delta) into a 16-bit shared tile for the dQ and dK
//                  MMAs; at the end dV (first) and dK (second) to HBM
//   warps 12..15 one thread per query row: dQ_part from TMEM (freeing its
//                  columns), then, once the tile's dK MMA (the last reader of
//                  its Q and dO) is done, staged in shared memory over the
//                  tile's Q and dO (128 x D fp32 is exactly their size), for
//                  the reducer (every key tile of a query row contributes to
//                  its dQ)
// A preprocessing kernel forms Delta, a final one converts the fp32 dQ
// (both in sdpa_bwd_prep.cuh).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "sdpa_kernel.cuh"

namespace sdpa {
namespace bwd {

constexpr int kThreads = 512;
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kReduceWarp = 2;
constexpr int kStatsWarp = 3;
constexpr int kSoftmaxWarp0 = 4;     // warps 4..11: two warpgroups, 64 queries each
constexpr int kDqWarp0 = 12;         // warps 12..15
// Register split: launched at 128 per thread (512 x 128 = 65536); warps 0..3
// drop to 80, the two softmax warpgroups and the dQ warpgroup rise to 144:
// 128 x 80 + 384 x 144 = 65536 (56 / 152 spilled).
constexpr uint32_t kRegsLow = 80;
constexpr uint32_t kRegsSoftmax = 144;
constexpr uint32_t kRegsDq = 144;
static_assert(128 * kRegsLow + 256 * kRegsSoftmax + 128 * kRegsDq <= kThreads * 128, "register split");
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSliceBytes = kBlockM * 128;   // 32 fp32 columns of a 128-row dQ tile

enum : unsigned int {
    kErrBwdWait = 0x400,             // + barrier id: a backward-pass wait timed out
};

struct Params {
    const float* lse;                // [B][Hq][Sq] natural log-sum-exp of the forward
    const float* delta;              // [B][Hq][Sq] dO_i . O_i
    float* dq_acc;                   // [B][Sq][Hq][D] fp32, zero on entry
    void* dK;                        // [B][Skv][Hkv][D] 16-bit
    void* dV;
    int B, Hq, Hkv, Sq, Skv, group;
    int n_qt, n_kt;                  // query / key tiles of 128
    int causal;
    float scale;
    float scale_log2;                // scale * log2(e)
};

struct BwdBarriers {
    uint64_t kv_full;
    uint64_t q_full[2];              // Q tile of stage s loaded
    uint64_t q_empty[2];             // Q tile of stage s free (its dQ slices reduced)
    uint64_t do_full[2];             // dO tile of stage s loaded
    uint64_t do_empty[2];            // dO tile of stage s free
    uint64_t s_full[2];              // S^T of tile it in TMEM: barrier it & 1
    uint64_t dp_full;                // dP^T in TMEM
    uint64_t p_ready;                // P^T packed in TMEM (both softmax warpgroups)
    uint64_t ds_ready;               // dS^T packed in TMEM and shared memory
    uint64_t dq_full;                // dQ_part of the tile in TMEM
    uint64_t dq_free;                // dQ_part read out of TMEM (its columns free for the next dP^T)
    uint64_t dk_done;                // the tile's dK MMA complete (its Q / dO stage may take dQ_part)
    uint64_t dkv_full;
    uint64_t stats_full[2];          // LSE2 / Delta buffer written (count 32)
    uint64_t dstage_full[2][4];      // dQ_part slice j staged over Q / dO stage s (count 128)
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// Shared memory: K, V (one tile each), Q and dO (two stages each), the dS^T
// tile for dQ (keys x 128 queries, 16-bit, two 64-query chunks with the
// 128-byte swizzle), LSE2 / Delta of the query tile in two buffers, barriers.
template <int D>
struct BwdLayout {
    static constexpr int kRowBytes = D * 2;
    static constexpr int kSwz = kRowBytes < 128 ? kRowBytes : 128;
    static constexpr int kChunks = kRowBytes / kSwz;
    static constexpr int kChunkBytes = kBlockM * kSwz;
    static constexpr int kTileBytes = kBlockM * kRowBytes;
    static constexpr int kSbo = 8 * kSwz;
    static constexpr uint32_t kSwzCode = (kSwz == 128) ? 2u : 4u;
    static constexpr int kSteps = kRowBytes / 32;                      // K = D MMAs: 16 elements each
    static constexpr int kOffK = 0;
    static constexpr int kOffV = kOffK + kTileBytes;
    static constexpr int kOffQ = kOffV + kTileBytes;                  // 2 stages
    static constexpr int kOffDO = kOffQ + 2 * kTileBytes;             // 2 stages
    static constexpr int kOffDS = kOffDO + 2 * kTileBytes;            // 128 x 128 x 2 bytes
    static constexpr int kDSChunkBytes = kBlockN * 128;               // 64 queries of every key row
    static constexpr int kOffStats = kOffDS + 2 * kDSChunkBytes;      // 2 x (LSE2[128], Delta[128])
    static constexpr int kOffBar = kOffStats + 2 * 2 * kBlockM * 4;
    // the dynamic shared memory is declared 1024-byte aligned (the 128-byte
    // swizzle needs it), so no alignment slack is added
    static constexpr int kSmemBytes = kOffBar + 256;
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
    // D = 64 leaves 128 columns free: S^T alternates between two regions, so
    // the next tile's S^T needs no wait for this tile's dV MMA
    static constexpr bool kTwoS = (D == 64);
    static constexpr uint32_t kColS2 = 384;
    static_assert(!kTwoS || kColDK + D <= kColS2, "second S^T region");
    static_assert(sizeof(BwdBarriers) <= 256, "barrier block");
    static_assert(D / 32 <= 4, "staging barriers: one per 32-column slice");
    static_assert(kColDK + D <= 512, "TMEM columns");
};


// The query tiles a CTA visits: for each head of its KV head's group, query
// tiles qt0 .. n_qt-1 (causal: qt0 = the CTA's key tile, the first query
// tile with a row that sees one of its keys; rows are top-left aligned).
__device__ __forceinline__ int bwd_qt0(const Params& p, int kt)
{
    return p.causal ? kt : 0;
}

template <int D, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
sdpa_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_dq, const Params p)
{
    using L = BwdLayout<D>;
    constexpr bool kOutBF16 = (KIND == sdpa::kBF16);
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (smem_u32(smem_raw) & 1023u) {
        // the layout relies on the declared alignment; never seen otherwise
        if (threadIdx.x == 0)
            atomicCAS(&g_sdpa_error, 0u, kErrBwdWait + 15);
        return;
    }
    uint8_t* smem = smem_raw;
    auto* bars = reinterpret_cast<BwdBarriers*>(smem + L::kOffBar);
    volatile int* abort = &bars->abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // this CTA: key tile kt of KV head hkv of batch b; key tiles in
    // ascending order over the grid, so under the causal mask the CTAs with
    // the most query tiles start first (longest first keeps the last wave
    // short)
    const int n_bg = p.B * p.Hkv;
    const int kt = blockIdx.x / n_bg;
    const int bg = blockIdx.x % n_bg;
    const int hkv = bg % p.Hkv;
    const int b = bg / p.Hkv;
    const int qt0 = bwd_qt0(p, kt);
    const int n_q = p.n_qt > qt0 ? p.n_qt - qt0 : 0;
    const int n_iter = n_q * p.group;            // (head, query tile) pairs, head-major

    const uint32_t sK = smem_u32(smem + L::kOffK);
    const uint32_t sV = smem_u32(smem + L::kOffV);
    const uint32_t sQ = smem_u32(smem + L::kOffQ);
    const uint32_t sDO = smem_u32(smem + L::kOffDO);
    const uint32_t sDS = smem_u32(smem + L::kOffDS);
    float* stats = reinterpret_cast<float*>(smem + L::kOffStats);      // [2][LSE2 128 | Delta 128]

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bars->kv_full), 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&bars->q_full[s]), 1);
            mbar_init(smem_u32(&bars->q_empty[s]), 1);
            mbar_init(smem_u32(&bars->do_full[s]), 1);
            mbar_init(smem_u32(&bars->do_empty[s]), 1);
        }
        mbar_init(smem_u32(&bars->s_full[0]), 1);
        mbar_init(smem_u32(&bars->s_full[1]), 1);
        mbar_init(smem_u32(&bars->dp_full), 1);
        mbar_init(smem_u32(&bars->p_ready), 256);          // both softmax warpgroups
        mbar_init(smem_u32(&bars->ds_ready), 256);
        mbar_init(smem_u32(&bars->dq_full), 1);
        mbar_init(smem_u32(&bars->dq_free), 128);
        mbar_init(smem_u32(&bars->dk_done), 1);
        mbar_init(smem_u32(&bars->dkv_full), 1);
        mbar_init(smem_u32(&bars->stats_full[0]), 32);
        mbar_init(smem_u32(&bars->stats_full[1]), 32);
        for (int s = 0; s < 2; ++s)
            for (int j = 0; j < 4; ++j)
                mbar_init(smem_u32(&bars->dstage_full[s][j]), 128);
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
            constexpr int kCe = L::kSwz / 2;                       // elements per chunk
            mbar_arrive_expect_tx(smem_u32(&bars->kv_full), 2 * L::kTileBytes);
            for (int c = 0; c < L::kChunks; ++c) {
                tma_load_4d(sK + c * L::kChunkBytes, &tm_k, smem_u32(&bars->kv_full), c * kCe, hkv, kt * kBlockN, b);
                tma_load_4d(sV + c * L::kChunkBytes, &tm_v, smem_u32(&bars->kv_full), c * kCe, hkv, kt * kBlockN, b);
            }
            int issued = 0;
            for (int it = 0; it < n_iter; ++it) {
                const int s = it & 1;
                // Q and dO of a stage are freed separately (the reducer reads
                // the dQ slices staged over Q first): Q, which S^T needs
                // first, is refilled as soon as it is free
                const int h = head_of(it), qt = qtile_of(it);
                if (it >= 2 &&
                    !wait_bar(smem_u32(&bars->q_empty[s]), ((it >> 1) & 1) ^ 1, abort, kErrBwdWait + 1))
                    break;
                mbar_arrive_expect_tx(smem_u32(&bars->q_full[s]), L::kTileBytes);
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_4d(sQ + s * L::kTileBytes + c * L::kChunkBytes, &tm_q, smem_u32(&bars->q_full[s]),
                                c * kCe, h, qt * kBlockM, b);
                ++issued;
                if (it >= 2 &&
                    !wait_bar(smem_u32(&bars->do_empty[s]), ((it >> 1) & 1) ^ 1, abort, kErrBwdWait + 12))
                    break;
                mbar_arrive_expect_tx(smem_u32(&bars->do_full[s]), L::kTileBytes);
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_4d(sDO + s * L::kTileBytes + c * L::kChunkBytes, &tm_do, smem_u32(&bars->do_full[s]),
                                c * kCe, h, qt * kBlockM, b);
                ++issued;
            }
            {
                // never leave the CTA with copies in flight: the last phase of
                // every slot (complete already in a normal run; after an
                // abort, the copies still landing)
                drain_wait(smem_u32(&bars->kv_full), 0);
                // issued counts the loads in order (Q of a tile, then its dO)
                for (int k = (issued > 4 ? issued - 4 : 0); k < issued; ++k) {
                    const int it = k >> 1;
                    drain_wait(smem_u32(&((k & 1) ? bars->do_full : bars->q_full)[it & 1]), (it >> 1) & 1);
                }
            }
        }
    } else if (warp == kMmaWarp) {
        // ============================ MMA issuer ============================
        if (lane == 0 && n_iter > 0) {
            constexpr uint32_t kFmt = kOutBF16 ? 1u : 0u;
            constexpr uint32_t id_s = idesc_make(kFmt, kBlockM, kBlockN, false);    // K-major A and B
            constexpr uint32_t id_o = idesc_make(kFmt, kBlockM, D, true);           // A in TMEM, B MN-major
            constexpr uint32_t id_q = idesc_make_amn(kFmt, kBlockM, D, true);       // A and B MN-major
            // descriptors as (hi, lo) halves: K-major use of a tile (LBO unused)
            // and MN-major use (LBO = the next 64-element chunk)
            const uint32_t hi = (uint32_t)(smem_desc(0, 16, L::kSbo, L::kSwzCode) >> 32);
            const uint32_t hi_ds = (uint32_t)(smem_desc(0, 16, 1024, 2u) >> 32);
            const uint32_t kmaj = 1u << 16;
            const uint32_t mnmaj = (uint32_t)(L::kChunkBytes >> 4) << 16;
            const uint32_t k_lo = (sK >> 4) | kmaj, k_mn = (sK >> 4) | mnmaj;
            const uint32_t v_lo = (sV >> 4) | kmaj;
            const uint32_t ds_lo = (sDS >> 4) | ((uint32_t)(L::kDSChunkBytes >> 4) << 16);   // MN-major use
            const uint32_t dsk_lo = (sDS >> 4) | kmaj;                                          // K-major use
            const uint32_t dp_t = tmem + L::kColDP;
            auto s_of = [&](int it) -> uint32_t { return tmem + ((L::kTwoS && (it & 1)) ? L::kColS2 : L::kColS); };
            const uint32_t dv_t = tmem + L::kColDV, dk_t = tmem + L::kColDK;
            // S^T = K Q^T (keys x queries, K = D) of tile `it` into cols 0..127
            auto issue_s = [&](int it) -> bool {
                const int s = it & 1;
                if (!wait_bar(smem_u32(&bars->q_full[s]), (it >> 1) & 1, abort, kErrBwdWait + 3))
                    return false;
                tc_fence_after_sync();
                const uint32_t q_lo = ((sQ + s * L::kTileBytes) >> 4) | kmaj;
#pragma unroll
                for (int kk = 0; kk < L::kSteps; ++kk) {
                    const uint32_t off = (uint32_t)(((kk * 32 / L::kSwz) * L::kChunkBytes + (kk * 32) % L::kSwz) >> 4);
                    mma_f16_ss(s_of(it), desc_join(hi, k_lo + off), desc_join(hi, q_lo + off), id_s, kk > 0);
                }
                mma_commit(smem_u32(&bars->s_full[it & 1]));
                return true;
            };
            bool ok = wait_bar(smem_u32(&bars->kv_full), 0, abort, kErrBwdWait + 2);
            if (ok)
                ok = issue_s(0);
            for (int it = 0; ok && it < n_iter; ++it) {
                const int s = it & 1;
                bool s_next = it + 1 >= n_iter;             // the next tile's S^T issued
                const uint32_t q_mn = ((sQ + s * L::kTileBytes) >> 4) | mnmaj;
                const uint32_t do_lo = ((sDO + s * L::kTileBytes) >> 4) | kmaj;
                const uint32_t do_mn = ((sDO + s * L::kTileBytes) >> 4) | mnmaj;
                // dP^T = V dO^T into cols 128..255, once the dQ warps have read the
                // last tile's dQ_part out of them
                if (it > 0 && !(ok = wait_bar(smem_u32(&bars->dq_free), (it - 1) & 1, abort, kErrBwdWait + 4)))
                    break;
                if (!(ok = wait_bar(smem_u32(&bars->do_full[s]), (it >> 1) & 1, abort, kErrBwdWait + 14)))
                    break;
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < L::kSteps; ++kk) {
                    const uint32_t off = (uint32_t)(((kk * 32 / L::kSwz) * L::kChunkBytes + (kk * 32) % L::kSwz) >> 4);
                    mma_f16_ss(dp_t, desc_join(hi, v_lo + off), desc_join(hi, do_lo + off), id_s, kk > 0);
                }
                mma_commit(smem_u32(&bars->dp_full));
                // D = 64: the next tile's S^T into the other region at once if
                // its Q has landed (that region's last readers, the last tile's
                // softmax and dV MMA, are done / issued)
                if (L::kTwoS && !s_next &&
                    mbar_test_wait(smem_u32(&bars->q_full[(it + 1) & 1]), ((it + 1) >> 1) & 1)) {
                    if (!(ok = issue_s(it + 1)))
                        break;
                    s_next = true;
                }
                // dV += P^T dO as soon as P^T is packed: 16 queries per step, P^T
                // from TMEM (8 columns per step: queries 0..63 in cols 0..31,
                // 64..127 in cols 64..95), dO MN-major
                if (!(ok = wait_bar(smem_u32(&bars->p_ready), it & 1, abort, kErrBwdWait + 5)))
                    break;
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < kBlockM / 16; ++kk) {
                    const uint32_t off = (uint32_t)((kk * 16 * L::kSwz) >> 4);
                    const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
                    const uint32_t col = (kk < 4) ? 8 * kk : 32 + 8 * kk;
                    mma_f16_ts(dv_t, s_of(it) + col, desc_join(hi, do_mn + off), id_o, acc);
                }
                // the next tile's S^T right after this dV MMA (the last reader of
                // cols 0..127) if its Q has landed: it runs while the softmax
                // forms dS^T, so the next P^T can start when this dS^T is done.
                // Otherwise after the dQ MMA, not to hold up dK and dQ.
                if (!s_next && mbar_test_wait(smem_u32(&bars->q_full[(it + 1) & 1]), ((it + 1) >> 1) & 1)) {
                    if (!(ok = issue_s(it + 1)))
                        break;
                    s_next = true;
                }
                // dQ_part = dS K first, into cols 128..128+D-1 (free once the
                // softmax has read dP^T): its read-out frees those columns for
                // the next dP^T.  A = dS (queries x keys) from the dS^T tile read
                // MN-major, 16 keys (rows of 128 bytes) per step; K MN-major.
                if (!(ok = wait_bar(smem_u32(&bars->ds_ready), it & 1, abort, kErrBwdWait + 10)))
                    break;
                tc_fence_after_sync();
#pragma unroll
                for (int kk = 0; kk < kBlockN / 16; ++kk) {
                    const uint32_t off_a = (uint32_t)((kk * 16 * 128) >> 4);
                    const uint32_t off_b = (uint32_t)((kk * 16 * L::kSwz) >> 4);
                    mma_f16_ss(dp_t, desc_join(hi_ds, ds_lo + off_a), desc_join(hi, k_mn + off_b), id_q, kk > 0);
                }
                mma_commit(smem_u32(&bars->dq_full));
                // dK += dS^T Q: A = the same dS^T tile read K-major (key rows,
                // 16 queries = 32 bytes per step, 64-query chunks), Q MN-major
#pragma unroll
                for (int kk = 0; kk < kBlockM / 16; ++kk) {
                    const uint32_t off_a = (uint32_t)(((kk / 4) * L::kDSChunkBytes + (kk % 4) * 32) >> 4);
                    const uint32_t off_b = (uint32_t)((kk * 16 * L::kSwz) >> 4);
                    const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
                    mma_f16_ss(dk_t, desc_join(hi_ds, dsk_lo + off_a), desc_join(hi, q_mn + off_b), id_o, acc);
                }
                mma_commit(smem_u32(&bars->dk_done));       // Q / dO of stage s: no MMA reads them any more
                if (!s_next && !(ok = issue_s(it + 1)))
                    break;
            }
            mma_commit(smem_u32(&bars->dkv_full));
            mma_commit(smem_u32(&bars->drain));
            drain_wait(smem_u32(&bars->drain), 0);
        }
      } else if (warp == kReduceWarp) {
        // ==================== dQ_part into the fp32 accumulator ==============
        if (lane == 0 && n_iter > 0) {
            tma_prefetch_map(&tm_dq);
            for (int it = 0; it < n_iter; ++it) {
                const int s = it & 1;
                const int h = head_of(it), qt = qtile_of(it);
                // each slice as soon as it is staged, those over Q first, then
                // those over dO: two bulk groups
                bool staged = true;
                for (int half = 0; staged && half < 2; ++half) {
                    for (int j = half * (D / 64); j < (half + 1) * (D / 64); ++j) {
                        if (!(staged = wait_bar(smem_u32(&bars->dstage_full[s][j]), (it >> 1) & 1, abort,
                                                kErrBwdWait + 13)))
                            break;
                        const uint32_t slice = (half == 0 ? sQ + (uint32_t)(j * kSliceBytes)
                                                          : sDO + (uint32_t)((j - D / 64) * kSliceBytes)) +
                                               (uint32_t)(s * L::kTileBytes);
                        tma_reduce_add_4d(&tm_dq, slice, 32 * j, h, qt * kBlockM, b);   // rows past Sq are clipped
                    }
                    bulk_commit_group();
                }
                if (!staged)
                    break;
                bulk_wait_group_read1();                    // Q of stage s may be refilled
                mbar_arrive(smem_u32(&bars->q_empty[s]));
                bulk_wait_group_read0();                    // and its dO
                mbar_arrive(smem_u32(&bars->do_empty[s]));
            }
            bulk_wait_group0();                             // the reductions have landed
        }
      } else if (warp == kStatsWarp) {
        // ====================== LSE2 / Delta of each tile =====================
        // Four query rows per lane into buffer it & 1: LSE2 = LSE log2(e)
        // (+inf past Sq: no weight) and Delta.  The buffer of tile it + 1 is
        // written once p_ready of tile it shows both softmax warpgroups done
        // with tile it - 1, its last readers; the wait is one tile ahead of
        // its use, and p_ready of tile it + 1 cannot come before this write.
        for (int it = 0; it < n_iter; ++it) {
            if (it > 0 &&
                !__all_sync(0xffffffffu, wait_bar(smem_u32(&bars->p_ready), (it - 1) & 1, abort, kErrBwdWait + 16)))
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
        // ==================== P^T and dS^T, one thread per key ===============
        const int sw = (warp - kSoftmaxWarp0) >> 2;         // query half of this warpgroup
        const int quarter = warp & 3;
        const int kr = quarter * 32 + lane;                 // key row of the tile (= TMEM lane)
        const int key = kt * kBlockN + kr;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const uint32_t dp_t = tmem + lane_addr + L::kColDP;
        const float c = p.scale_log2;
        const bool key_ok = key < p.Skv;
        bool ok = true;
        for (int it = 0; ok && it < n_iter; ++it) {
            ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->s_full[it & 1]), (it >> 1) & 1, abort,
                                                  kErrBwdWait + 6));
            const uint32_t s_t = tmem + lane_addr + ((L::kTwoS && (it & 1)) ? L::kColS2 : L::kColS);
            if (ok)
                ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->stats_full[it & 1]), (it >> 1) & 1, abort,
                                                      kErrBwdWait + 9));
            if (!ok)
                break;
            tc_fence_after_sync();
            const float4* l2v = reinterpret_cast<const float4*>(stats + (it & 1) * 2 * kBlockM);
            const float4* dlv = l2v + kBlockM / 4;
            // top-left causal: this key is visible to query q iff key <= q;
            // keys past Skv are visible to none
            const int first_q = !key_ok ? (1 << 30) : (p.causal ? key - qtile_of(it) * kBlockM : -1);
            // phase 1, from S^T alone: P^T, packed over this warpgroup's own
            // S^T columns (already read; the other warpgroup may not have read
            // its own yet): queries 64 sw + 32 chh .. +31 in cols 64 sw + 16 chh ..
            float pf[2][32];
#pragma unroll
            for (int chh = 0; chh < 2; ++chh) {             // 32 queries per chunk, two per warpgroup
                const int ch = 2 * sw + chh;
                uint32_t sv[32];
                tmem_ld32_wait(s_t + 32 * ch, sv);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 l4 = l2v[8 * ch + i];
                    const float lq[4] = {l4.x, l4.y, l4.z, l4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int q = 32 * ch + 4 * i + e;
                        pf[chh][4 * i + e] =
                            q >= first_q ? ex2_approx(__uint_as_float(sv[4 * i + e]) * c - lq[e]) : 0.f;
                    }
                    pk[2 * i] = pack2<kOutBF16>(pf[chh][4 * i], pf[chh][4 * i + 1]);
                    pk[2 * i + 1] = pack2<kOutBF16>(pf[chh][4 * i + 2], pf[chh][4 * i + 3]);
                }
                tmem_st16(s_t + 64 * sw + 16 * chh, pk);
            }
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(smem_u32(&bars->p_ready));          // dV += P^T dO can start
            // phase 2, once dP^T is there: dS^T = scale P^T (dP^T - Delta),
            // packed over the warpgroup's own dP^T columns and into the
            // shared tile for dQ
            ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->dp_full), it & 1, abort, kErrBwdWait + 11));
            if (!ok)
                break;
            tc_fence_after_sync();
#pragma unroll
            for (int chh = 0; chh < 2; ++chh) {
                const int ch = 2 * sw + chh;
                uint32_t dv[32];
                tmem_ld32_wait(dp_t + 32 * ch, dv);
                uint32_t dk[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float4 d4 = dlv[8 * ch + i];
                    const float dq[4] = {d4.x, d4.y, d4.z, d4.w};
                    float ds[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        ds[e] = pf[chh][4 * i + e] * p.scale * (__uint_as_float(dv[4 * i + e]) - dq[e]);
                    dk[2 * i] = pack2<kOutBF16>(ds[0], ds[1]);
                    dk[2 * i + 1] = pack2<kOutBF16>(ds[2], ds[3]);
                }
                // dS^T row for the dQ and dK MMAs: queries 32ch .. 32ch+31 are 16-byte units
                // 4(ch&1) .. +3 of 64-query chunk ch/2 (= sw), 128-byte swizzle
                const uint32_t row_base = sDS + sw * L::kDSChunkBytes + kr * 128;
#pragma unroll
                for (int uu = 0; uu < 4; ++uu) {
                    const int u = 4 * chh + uu;
                    st_shared_v4(row_base + (uint32_t)((u ^ (kr & 7)) << 4), dk[4 * uu], dk[4 * uu + 1],
                                 dk[4 * uu + 2], dk[4 * uu + 3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before_sync();
            mbar_arrive(smem_u32(&bars->ds_ready));
        }
        // ---- dK, dV of this key (dK carries the scale already, through dS) ----
        // The wait and the TMEM loads are warp-wide (every lane takes part);
        // only keys below Skv store.
        if (ok && n_iter > 0) {
            ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->dkv_full), 0, abort, kErrBwdWait + 7));
            tc_fence_after_sync();
        }
        if (ok) {
            const int64_t row_off = (((int64_t)b * p.Skv + key) * p.Hkv + hkv) * D;
            {
                const int which = sw;                       // first warpgroup dV, second dK
                uint16_t* dst = reinterpret_cast<uint16_t*>(which ? p.dK : p.dV) + row_off;
                const uint32_t col = which ? L::kColDK : L::kColDV;
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc) {
                    uint32_t r[32];
                    if (n_iter > 0) {
                        tmem_ld32_wait(tmem + lane_addr + col + 32 * cc, r);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            r[i] = 0u;                      // no query sees this key
                    }
                    if (key_ok) {
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            reinterpret_cast<uint4*>(dst + 32 * cc)[v] = make_uint4(
                                pack2<kOutBF16>(__uint_as_float(r[8 * v]), __uint_as_float(r[8 * v + 1])),
                                pack2<kOutBF16>(__uint_as_float(r[8 * v + 2]), __uint_as_float(r[8 * v + 3])),
                                pack2<kOutBF16>(__uint_as_float(r[8 * v + 4]), __uint_as_float(r[8 * v + 5])),
                                pack2<kOutBF16>(__uint_as_float(r[8 * v + 6]), __uint_as_float(r[8 * v + 7])));
                    }
                }
            }
        }
    } else if (warp >= kDqWarp0) {
        regs_acquire<kRegsDq>();
        // ================== dQ_part into the fp32 accumulator ================
        const int quarter = warp & 3;
        const int qr = quarter * 32 + lane;                 // query row of the tile (= TMEM lane)
        const uint32_t src = tmem + ((uint32_t)(quarter * 32) << 16) + L::kColDP;   // dQ_part
        bool ok = true;
        for (int it = 0; ok && it < n_iter; ++it) {
            ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->dq_full), it & 1, abort, kErrBwdWait + 8));
            if (!ok)
                break;
            tc_fence_after_sync();
            // all D columns out of TMEM first, so the next tile's dP MMA can
            // take the columns while this tile's dQ is reduced into HBM
            uint32_t r[D];
#pragma unroll
            for (int c = 0; c < D / 32; ++c)
                tmem_ld32_wait(src + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * c]));
            tc_fence_before_sync();
            mbar_arrive(smem_u32(&bars->dq_free));
            // staged for the reducer over Q / dO stage s once the tile's dK
            // MMA, their last reader, has completed: 32-column slices of 128
            // rows x 128 bytes with the 128-byte swizzle, slices 0 .. D/64-1
            // over Q and the rest over dO
            ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->dk_done), it & 1, abort, kErrBwdWait + 17));
            if (!ok)
                break;
            const int s = it & 1;
#pragma unroll
            for (int j = 0; j < D / 32; ++j) {
                const uint32_t slice = (j < D / 64 ? sQ + (uint32_t)(j * kSliceBytes)
                                                   : sDO + (uint32_t)((j - D / 64) * kSliceBytes)) +
                                       (uint32_t)(s * L::kTileBytes);
                const uint32_t row = slice + (uint32_t)(qr * 128);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    st_shared_v4(row + (uint32_t)((u ^ (qr & 7)) << 4), r[32 * j + 4 * u], r[32 * j + 4 * u + 1],
                                 r[32 * j + 4 * u + 2], r[32 * j + 4 * u + 3]);
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&bars->dstage_full[s][j]));   // the reducer may start on it
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

}  // namespace bwd
}  // namespace sdpa
