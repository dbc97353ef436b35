// sdpa_kernel.cuh -- fused attention forward pass for sm_103a.
//
// Computes O = softmax(Q K^T * scale [+ causal mask]) V, the definition in the
// codelab "Attention on GPU (cuDNN and TransformerEngine)", section 1 ("How
// attention works"), in one pass over the keys with a running max and sum
// (online softmax), so the Sq x Skv score matrix never leaves the chip -- the
// tiling that section 8 ("Run benchmarks", sequence sweep) credits fused
// kernels with.
//
// Persistent kernel: one CTA per SM walks a static list of work units.  A
// unit is 256 query rows (two 128-row Q tiles, t = 0, 1) of one (batch,
// query head); both tiles share every K/V tile the producer brings in.
// Warp roles (12 warps):
//   warps 0..3   softmax warpgroup for Q tile 0
//   warps 4..7   softmax warpgroup for Q tile 1
//   warp 8       TMA producer: Q tiles, then K_j / V_j into shared-memory rings
//   warps 9, 10  tcgen05 issue of O_t += P_t V_j for Q tile 0 / 1
//   warp 11      tcgen05 issue of every S_t = Q_t K_j^T
// A second instance (QT = 1, 16-bit kinds at D <= 64, small problems) runs
// two CTAs per SM with units of one Q tile: 8 warps (softmax 0..3, producer
// 4, P V issue 5, S issue 7), half the TMEM columns and ~100 KB of shared
// memory each; see Roles below.
// Both Q tiles take turns in one TMEM S region.  P_t never overwrites S: the
// 16-bit P_t has its own TMEM columns, the E4M3 P_t sits in shared memory
// (and the tensor core sums its rows, P_t times a tile of ones).  So S_t(j+1)
// is computed while the softmax works on S_t(j), and each softmax warpgroup
// runs from key tile to key tile without waiting for its P V.
// Each softmax thread owns one query row: it reads its S row from TMEM, masks
// only the diagonal / tail tile, keeps the running max m (exp2 domain) and
// the sum l in fp32, forms P = exp2(S*c - m), and rescales its O row (and l)
// only when m grows by more than 8 (a factor 256; 3 for E4M3; P and l stay
// exact relative to the m actually used).  After the unit's last tile it
// reads O_t, releases the accumulator for the next unit, and stores O / l to
// HBM.
//
// Layout: Q, O are [B][Sq][Hq][D] and K, V are [B][Skv][Hkv][D] (section 3,
// "Create Q, K and V test arrays": (B, T, N, H)).  Query head hq reads KV head
// hq / (Hq / Hkv) (section 9, "Compare MHA, GQA and MQA"); nothing is
// replicated.  Causal masking keeps the lower triangle (section 7, "Add causal
// masking"): row i sees keys 0..i; key tiles wholly above the diagonal are
// skipped.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace sdpa {

constexpr int kBlockM = 128;         // query rows per Q tile (= TMEM lanes)
constexpr int kBlockN = 128;         // keys per K/V tile
// Warp roles for QT Q tiles per CTA.  QT = 2 (the standard pass, one CTA
// per SM): warps 0..7 are two softmax warpgroups, warp 8 the TMA producer,
// warps 9 / 10 the P V issuers of Q tile 0 / 1, warp 11 the S issuer; both
// Q tiles read every K / V tile the CTA loads.  QT = 1 (16-bit kinds at
// D <= 64, two CTAs per SM): warps 0..3 softmax, 4 producer, 5 P V issuer,
// 7 S issuer (warp 6 idles); the two CTAs of an SM run independent units of
// one Q tile each, so a unit's epilogue overlaps the other CTA's key tiles.
template <int QT>
struct Roles {
    static_assert(QT == 1 || QT == 2, "Q tiles per CTA");
    static constexpr int kUnitRows = QT * kBlockM;
    static constexpr int kThreads = 128 * QT + 128;
    static constexpr int kProducerWarp = 4 * QT;
    static constexpr int kMmaWarp = 4 * QT + 1;      // P V issue for Q tile 0 (+ 1: Q tile 1)
    static constexpr int kSMmaWarp = 4 * QT + 3;     // S issue
    static constexpr int kCtasPerSm = 3 - QT;
    // Register split: launched at 168 per thread (QT = 2: 384 x 168 = 64512)
    // or 128 (QT = 1: two CTAs of 256 x 128); the producer warpgroup drops to
    // 104 / 64 and the softmax warpgroups rise to 192.
    static constexpr uint32_t kLaunchRegs = (QT == 2) ? 168u : 128u;
    static constexpr uint32_t kRegsProducer = (QT == 2) ? 104u : 64u;
    static constexpr uint32_t kRegsSoftmax = 192;
    static_assert(128 * kRegsProducer + 128 * QT * kRegsSoftmax <= kThreads * kLaunchRegs,
                  "register split exceeds the launch budget");
    static_assert(kThreads * kLaunchRegs * kCtasPerSm <= 65536, "register file");
};
// the standard pass's unit (also the packed decode pass's)
constexpr int kUnitRows = Roles<2>::kUnitRows;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s per barrier wait
constexpr float kRescaleThreshold = 8.0f;          // log2 units: rescale O when m grows by > 2^8
// E4M3 P: rescale when m grows by > 2^3 and store P * 56, so that
// P * 56 <= 2^3 * 56 = 448, the largest finite E4M3 value.
constexpr float kRescaleThresholdFP8 = 3.0f;
constexpr float kLog2P8Scale = 5.807354922057604f;  // log2(56)
constexpr float kLn2 = 0.6931471805599453f;

// Device error word: 0 = no error; otherwise the first failure recorded by any
// CTA (see the codes below).  Read and cleared by the host through the C-ABI.
__device__ unsigned int g_sdpa_error = 0;

#ifdef SDPA_WAIT_TEST
// Test build only (compiled with -DSDPA_WAIT_TEST into a separate library):
// the wait limit and a K-ring position whose copy the forward producer leaves
// out, both set from the host, so that a test can make a bounded wait run out
// on the GPU without any fault.  The product library has neither.
__device__ uint64_t g_test_wait_limit_ns = kWaitLimitNs;
__device__ int g_test_withhold_k = -1;
__device__ __forceinline__ uint64_t wait_limit_ns() { return g_test_wait_limit_ns; }
#else
__device__ __forceinline__ constexpr uint64_t wait_limit_ns() { return kWaitLimitNs; }
#endif

// Polls of the S-issue count before a P V MMA is issued anyway (~30 cycles
// each): about twice the longest S_t(j+1) delay seen in clock traces.
constexpr int kOrderSpins = 256;

enum : unsigned int {
    kErrWaitLoad = 0x100,            // + barrier id: producer wait timed out
    kErrWaitMma = 0x200,             // + barrier id: MMA issuer wait timed out
    kErrWaitSoftmax = 0x300,         // + barrier id: softmax wait timed out
};

struct Params {
    void* O;
    long long o_sb, o_ss, o_sh;      // O strides in elements (batch, sequence, head); D is contiguous
    float* lse;                      // [B][Hq][Sq] log-sum-exp of each row's scores, or null
    int B, Hq, Hkv, Sq, Skv;
    int group;                       // Hq / Hkv
    int n_units;                     // B * Hq * n_pairs
    int n_pairs;                     // ceil(Sq / 256)
    int n_ktiles;                    // ceil(Skv / 128)
    int causal;
    float scale_log2;                // scale * log2(e) (* descale_q * descale_k for E4M3)
    float out_scale;                 // descale_v for E4M3, else 1
    // packed (decode) mode only: key tiles per split, splits, and the split
    // results (null with one split): per packed row (b, h, s) and split, O / l
    // in fp32 [B][Hq][Sq][n_splits][D] and the LSE [B][Hq][Sq][n_splits]
    int tiles_per_split;
    int n_splits;
    float* part_o;
    float* part_lse;
};

// Element kinds of Q, K and V.
enum Kind : int { kBF16 = 0, kFP16 = 1, kE4M3 = 2 };

// Shared-memory and TMEM layout for head dimension D and element kind KIND.
// A Q / K / V tile is 128 rows of D elements; TMA writes it as column blocks
// ("chunks") of kSwz bytes per row with the matching hardware swizzle
// (128-byte, or 64-byte when a row holds only 64 bytes).
template <int D, int KIND, int QT = 2>
struct Layout {
    static_assert(D == 32 || D == 64 || D == 128, "head dimension");
    static_assert(QT == 2 || (KIND != kE4M3 && D <= 64), "one Q tile per CTA: 16-bit kinds, D <= 64");
    static_assert(D != 32 || KIND != kE4M3, "E4M3 needs rows of at least 64 bytes");
    static constexpr int kEsize = (KIND == kE4M3) ? 1 : 2;
    static constexpr int kRowBytes = D * kEsize;
    static constexpr int kSwz = kRowBytes < 128 ? kRowBytes : 128;     // swizzle span in bytes
    static constexpr int kChunks = kRowBytes / kSwz;
    static constexpr int kChunkBytes = kBlockM * kSwz;
    static constexpr int kTileBytes = kBlockM * kRowBytes;              // one Q, K or V tile
    static constexpr int kSbo = 8 * kSwz;                              // 8-row group stride
    static constexpr uint32_t kSwzCode = (kSwz == 128) ? 2u : 4u;        // descriptor swizzle field
    static constexpr int kSSteps = kRowBytes / 32;                     // S MMAs: 32 bytes of K each
    static constexpr int kKeysPerStep = 32 / kEsize;                   // P V MMAs: 16 (16-bit) or 32 (8-bit) keys
    static constexpr int kPVSteps = kBlockN / kKeysPerStep;
    // 16-bit D = 128 keeps 2 K stages, E4M3 D = 128 3 V stages, so that the
    // output staging below fits; one Q tile per CTA keeps 2 + 2 stages of
    // 16 KB tiles, so that two CTAs fit on an SM
    static constexpr int kStagesK = (kTileBytes >= 32768 || (QT == 1 && kTileBytes >= 16384)) ? 2 : 4;
    static constexpr int kStagesV = (kTileBytes >= 32768 || (QT == 1 && kTileBytes >= 16384)) ? 2
                                    : (KIND == kE4M3 && D == 128)                                 ? 3
                                                                                                  : 4;
    static constexpr int kOffQ = 0;                                    // Q tile 0 (, Q tile 1)
    static constexpr int kOffK = kOffQ + QT * kTileBytes;
    static constexpr int kOffV = kOffK + kStagesK * kTileBytes;
    // E4M3: P_t lives in shared memory (128 rows x 128 keys, one byte each,
    // 128-byte swizzled rows), one tile per Q tile; 16-bit P stays in TMEM.
    // E4M3 also keeps a 16 x 128 tile of ones (E4M3 1.0 = 0x38): the MMA
    // P_t x ones sums each row of P into TMEM.
    static constexpr int kPTileBytes = kBlockM * kBlockN;
    static constexpr int kOnesBytes = 16 * kBlockN;
    static constexpr int kOffP = kOffV + kStagesV * kTileBytes;
    static constexpr int kOffOnes = kOffP + 2 * kPTileBytes;
    // Output staging: each softmax warp writes its 32 rows of O (16-bit,
    // bf16 for E4M3 inputs) here, one swizzle span (kOSwz bytes) of every row
    // per pass, and a TMA tensor store moves them to HBM in whole lines.
    static constexpr int kORowBytes = D * 2;
    static constexpr int kOSwz = kORowBytes < 128 ? kORowBytes : 128;
    static constexpr int kOPasses = kORowBytes / kOSwz;
    static constexpr int kOWarpBytes = 32 * kOSwz;
    static constexpr int kOffO = (KIND == kE4M3) ? kOffOnes + kOnesBytes : kOffP;
    static_assert(kOffO % 1024 == 0, "output staging must sit on a swizzle-atom boundary");
    static constexpr int kOffBar = kOffO + 4 * QT * kOWarpBytes;
    static constexpr int kBarBytes = 1024;
    static constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;     // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory budget");
    static_assert(QT == 2 || 2 * (kSmemBytes + 1024) <= 233472, "two CTAs per SM");
    // TMEM columns (512, or 256 with one Q tile per CTA).  O_t takes the last
    // QT x D columns.  Both Q tiles take turns in one S region (columns
    // 0..127), except for 16-bit kinds at D = 64 with two Q tiles, where each
    // has its own (128 t).  (E4M3 keeps the shared region at D = 64 too: it
    // measured faster there, the shared region staggering the two softmax
    // warpgroups.)  After the S columns: 16-bit P_t (64 columns each, two
    // values per column) or, for E4M3 (P in shared memory), the row sums l_t
    // (16 columns each, all equal).
    static constexpr bool kSharedS = (D > 64) || (KIND == kE4M3) || (QT == 1);
    static constexpr uint32_t kTmemCols = (QT == 2) ? 512u : 256u;
    static constexpr uint32_t kAfterS = kSharedS ? 128u : 256u;
    __host__ __device__ static constexpr uint32_t tmem_s(int t) { return kSharedS ? 0u : 128u * t; }
    __host__ __device__ static constexpr uint32_t tmem_p(int t) { return kAfterS + 64u * t; }  // 16-bit kinds
    __host__ __device__ static constexpr uint32_t tmem_l(int t) { return kAfterS + 16u * t; }  // E4M3
    __host__ __device__ static constexpr uint32_t tmem_o(int t)
    {
        return kTmemCols - (uint32_t)(QT * D) + (uint32_t)D * t;
    }
    static_assert(kAfterS + 64u * QT <= kTmemCols - (uint32_t)(QT * D), "TMEM columns overlap");
};

template <int NK, int NV>
struct Barriers {
    uint64_t q_full[2];
    uint64_t q_empty[2];
    uint64_t k_full[NK];
    uint64_t k_empty[NK];
    uint64_t v_full[NV];
    uint64_t v_empty[NV];
    uint64_t s_full[2];
    uint64_t p_full[2];
    uint64_t o_full[2];
    uint64_t o_empty[2];
    uint64_t s_free[2];              // S_t read out of the S region (count 128)
    uint64_t pv_done[2];             // P_t V_j complete (P_t buffer free, O_t current)
    uint64_t drain[3];               // one per MMA-issuing thread
    uint32_t s_issued[2];            // S_t MMAs issued so far (a count, written by the S issuer)
    uint32_t tmem_base;
    int abort;
};

// Bounded wait: gives up after kWaitLimitNs (2 s), records `code` in the device
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
        if (global_timer_ns() - t0 > wait_limit_ns()) {
            *abort = 1;
            atomicCAS(&g_sdpa_error, 0u, code);
            return false;
        }
    }
}

// Waits without recording an error (used only to drain in-flight work after
// an abort).
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity) && global_timer_ns() - t0 < wait_limit_ns()) {
    }
}

// Two floats -> two 16-bit values (round to nearest even), lo in the low half.
template <bool kToBF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi)
{
    if constexpr (kToBF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

// Work unit -> (b, hq, pair).  Causal units are ordered heaviest first (the
// last query rows see the most keys).
struct Unit {
    int b, hq, hkv, pair;
    int n;                           // key tiles loaded for the unit: kv0 .. kv0 + n - 1
    int kv0;
    int split;                       // packed mode: which key range
    int n_kv[2];                     // key tiles visited by Q tile 0 / 1 (the first n_kv[t]; 0 = tile unused)
    // n_kv[t] for a t known only at run time, as a select: an indexed read
    // would put the struct in local memory (measured: FP8 forward +1.6 %,
    // causal MQA S=512 +3.6 %)
    __device__ __forceinline__ int kv(int t) const { return t ? n_kv[1] : n_kv[0]; }
};

// Packed (decode) mode: the Hq / Hkv = G query heads that read one KV head are
// stacked into the M rows of a Q tile, row r = s * G + h (query position s,
// head h of the group), so a K/V tile serves every head of the group at once;
// the key range may be split over several units.  Non-causal only.
// Unit u -> (KV head, batch, packed-row pair, split), KV head fastest.
template <bool kPacked, int QT = 2>
__device__ __forceinline__ Unit decode_unit(const Params& p, int u)
{
    Unit w;
    if constexpr (kPacked) {
        w.hkv = u % p.Hkv;
        int rest = u / p.Hkv;
        w.b = rest % p.B;
        rest /= p.B;
        w.pair = rest % p.n_pairs;
        w.split = rest / p.n_pairs;
        w.hq = w.hkv * p.group;
        w.kv0 = w.split * p.tiles_per_split;
        w.n = min(p.n_ktiles - w.kv0, p.tiles_per_split);
        const int rows = p.Sq * p.group;                   // packed rows of one (b, KV head)
        w.n_kv[0] = w.n;                                    // the pair exists, so tile 0 has rows
        w.n_kv[1] = (w.pair * kUnitRows + kBlockM < rows) ? w.n : 0;
        return w;
    }
    w.split = 0;
    w.kv0 = 0;
    const int bh_count = p.B * p.Hq;
    w.pair = u / bh_count;
    if (p.causal)
        w.pair = p.n_pairs - 1 - w.pair;
    const int bh = u % bh_count;
    w.b = bh / p.Hq;
    w.hq = bh % p.Hq;
    w.hkv = w.hq / p.group;
    if constexpr (QT == 1) {
        // one Q tile (w.pair is its index): causal rows of tile i see keys
        // below 128 (i + 1)
        w.n_kv[0] = p.causal ? min(p.n_ktiles, w.pair + 1) : p.n_ktiles;
        w.n_kv[1] = 0;
        w.n = w.n_kv[0];
        return w;
    }
    if (p.causal) {
        w.n_kv[0] = min(p.n_ktiles, 2 * w.pair + 1);
        w.n_kv[1] = min(p.n_ktiles, 2 * w.pair + 2);
    } else {
        w.n_kv[0] = w.n_kv[1] = p.n_ktiles;
    }
    w.n = w.n_kv[1];                 // tile 1 visits at least as many key tiles as tile 0
    return w;
}

// Static schedule: CTA c takes, in round r, unit r*G + c (r even) or
// r*G + G-1-c (r odd), G = gridDim.x.  With units sorted heaviest first this
// zig-zag pairs heavy and light causal units on every CTA.  Returns -1 when
// the CTA has no unit in round r (only possible in the last round) and -2
// once the rounds are exhausted.
__device__ __forceinline__ int unit_of_round(const Params& p, int r)
{
    const int G = gridDim.x;
    const int base = r * G;
    if (base >= p.n_units)
        return -2;
    const int u = base + ((r & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
    return u < p.n_units ? u : -1;
}

// Shared-memory descriptor from its two 32-bit halves.  The high half (SBO,
// version, swizzle) is the same for every operand of a kind; the low half
// holds the start address and LBO, so each MMA's descriptor is one 32-bit add
// away from a per-tile base.
__device__ __forceinline__ uint64_t desc_join(uint32_t hi, uint32_t lo)
{
    return ((uint64_t)hi << 32) | (uint64_t)lo;
}

// MMA issue.  P_t never aliases S (16-bit P has its own TMEM columns, E4M3 P
// sits in shared memory), so the next S needs only that the softmax has read
// the previous one out of TMEM, not that P_t V_j has run: S_t(j+1) is
// computed while the softmax works on S_t(j), and each softmax warpgroup
// goes from one key tile to the next without waiting for its P V.  Both Q
// tiles take turns in one S region.
//
// Three issuing threads: thread 0 of warp 11 issues every S, in region order
// S_0(0), S_1(0), S_0(1), S_1(1), ... (tile 0 drops out after its last causal
// key tile); thread 0 of warp 9 / 10 issues P_t V_j for Q tile 0 / 1.  The S
// thread waits, before each S, for the softmax of the previous S's tile to
// have read it (s_free[t]); as it waits for every S in order, no s_free
// barrier can be two phases away from the phase it waits for.

// Descriptors as (hi, lo) halves.  Q and K tiles are K-major and swizzled:
// one MMA takes 32 bytes of the row (16 bf16/fp16 or 32 E4M3 elements), which
// moves 32 bytes inside a swizzle chunk; chunks are kChunkBytes apart and
// 8-row groups kSbo apart.  The V tile is MN-major (D contiguous): a step of
// kKeysPerStep keys is kKeysPerStep rows of kSwz bytes, the next chunk of D
// columns kChunkBytes further (LBO).  The E4M3 P tile and the ones tile have
// 128-byte rows: one 128-byte swizzle span, 8-row groups 1024 bytes apart.
template <int D, int KIND, bool kPacked, int NK, int NV, int QT>
__device__ __forceinline__ void mma_issue_s(const Params& p, Barriers<NK, NV>* bars, volatile int* abort,
                                            uint32_t tmem, uint32_t sQ, uint32_t sK)
{
    using L = Layout<D, KIND, QT>;
    constexpr uint32_t kFmt = (KIND == kBF16) ? 1u : 0u;          // bf16 / f16 / E4M3
    constexpr uint32_t idesc_s = idesc_make(kFmt, kBlockM, kBlockN, false);
    constexpr uint32_t kTileUnits = L::kTileBytes >> 4;
    const uint32_t desc_hi = (uint32_t)(smem_desc(0, 16, L::kSbo, L::kSwzCode) >> 32);
    const uint32_t k_lo0 = (sK >> 4) | (1u << 16);
    uint32_t ck = 0;                     // K ring position
    uint32_t ns[2] = {0, 0};             // S tiles issued per Q tile
    int prev = -1;                       // Q tile of the last S issued
    uint32_t ua[2] = {0, 0};             // units in which Q tile 0 / 1 took part
    bool ok = true;
    for (int r = 0; ok; ++r) {
        const int u = unit_of_round(p, r);
        if (u == -2)
            break;
        if (u < 0)
            continue;
        const Unit w = decode_unit<kPacked, QT>(p, u);
        const int n = w.n;
        for (int j = 0; ok && j < n; ++j) {
            ok = wait_bar(smem_u32(&bars->k_full[ck % NK]), (ck / NK) & 1, abort, kErrWaitMma + 3);
            for (int t = 0; ok && t < 2; ++t) {
                if (j >= w.n_kv[t])
                    continue;
                if (j == 0)
                    ok = wait_bar(smem_u32(&bars->q_full[t]), ua[t] & 1, abort, kErrWaitMma + 1 + t);
                // the previous S in this region has been read out of it: the
                // last S of either tile (shared region) or of this tile
                const int pt = L::kSharedS ? prev : (ns[t] > 0 ? t : -1);
                if (ok && pt >= 0)
                    ok = wait_bar(smem_u32(&bars->s_free[pt]), (ns[pt] - 1) & 1, abort, kErrWaitMma + 12 + pt);
                if (!ok)
                    break;
                tc_fence_after_sync();
                const uint32_t q_lo = ((sQ + t * L::kTileBytes) >> 4) | (1u << 16);
                const uint32_t k_lo = k_lo0 + (ck % NK) * kTileUnits;
#pragma unroll
                for (int kk = 0; kk < L::kSSteps; ++kk) {
                    const uint32_t off = (uint32_t)(((kk * 32 / L::kSwz) * L::kChunkBytes + (kk * 32) % L::kSwz) >> 4);
                    const uint32_t s_tmem = tmem + L::tmem_s(t);
                    if constexpr (KIND == kE4M3)
                        mma_f8_ss(s_tmem, desc_join(desc_hi, q_lo + off), desc_join(desc_hi, k_lo + off), idesc_s,
                                  kk > 0);
                    else
                        mma_f16_ss(s_tmem, desc_join(desc_hi, q_lo + off), desc_join(desc_hi, k_lo + off), idesc_s,
                                   kk > 0);
                }
                mma_commit(smem_u32(&bars->s_full[t]));
                if (j == w.n_kv[t] - 1)
                    mma_commit(smem_u32(&bars->q_empty[t]));
                ++ns[t];
                *reinterpret_cast<volatile uint32_t*>(&bars->s_issued[t]) = ns[t];   // after the MMAs
                prev = t;
            }
            if (!ok)
                break;
            mma_commit(smem_u32(&bars->k_empty[ck % NK]));
            ++ck;
        }
        for (int t = 0; t < 2; ++t)
            ua[t] += (w.n_kv[t] > 0) ? 1u : 0u;
    }
    // every MMA this thread issued completes before TMEM is released
    mma_commit(smem_u32(&bars->drain[2]));
    drain_wait(smem_u32(&bars->drain[2]), 0);
}

// O_t (+)= P_t V_j for Q tile t, kKeysPerStep keys per MMA.  16-bit P_t is
// read from its TMEM columns (8 columns per step of 16 keys).  E4M3 P_t
// (K-major, keys contiguous) comes from shared memory, and l_t (+)= P_t x
// ones.  Every P V thread (QT of them) releases every V slot of the unit
// (barrier count QT), tile 0 also the causal key tile it does not visit.
template <int D, int KIND, bool kPacked, int NK, int NV, int QT>
__device__ __forceinline__ void mma_issue_pv(const Params& p, Barriers<NK, NV>* bars, volatile int* abort,
                                             uint32_t tmem, uint32_t sV, uint32_t sP, uint32_t sOnes, int t)
{
    using L = Layout<D, KIND, QT>;
    constexpr bool kFP8 = (KIND == kE4M3);
    constexpr uint32_t kFmt = (KIND == kBF16) ? 1u : 0u;
    constexpr uint32_t idesc_o = idesc_make(kFmt, kBlockM, D, true);
    constexpr uint32_t idesc_l = idesc_make(kFmt, kBlockM, 16, false);
    constexpr uint32_t kTileUnits = L::kTileBytes >> 4;
    const uint32_t p_tmem = tmem + L::tmem_p(t);
    const uint32_t o_tmem = tmem + L::tmem_o(t);
    const uint32_t l_tmem = tmem + L::tmem_l(t);
    const uint32_t desc_hi = (uint32_t)(smem_desc(0, 16, L::kSbo, L::kSwzCode) >> 32);
    const uint32_t p_hi = (uint32_t)(smem_desc(0, 16, 1024, 2u) >> 32);
    const uint32_t v_lo0 = (sV >> 4) | ((uint32_t)(L::kChunkBytes >> 4) << 16);
    const uint32_t p_lo = ((sP + t * L::kPTileBytes) >> 4) | (1u << 16);
    const uint32_t ones_lo = (sOnes >> 4) | (1u << 16);
    uint32_t cv = 0;                     // V ring position
    uint32_t npv = 0;                    // P V groups issued
    uint32_t units = 0;                  // units in which this Q tile took part
    bool ok = true;
    for (int r = 0; ok; ++r) {
        const int u = unit_of_round(p, r);
        if (u == -2)
            break;
        if (u < 0)
            continue;
        const Unit w = decode_unit<kPacked, QT>(p, u);
        const int n = w.n;
        const int nt = w.kv(t);
        for (int j = 0; ok && j < n; ++j, ++cv) {
            ok = wait_bar(smem_u32(&bars->v_full[cv % NV]), (cv / NV) & 1, abort, kErrWaitMma + 5);
            if (!ok)
                break;
            if (j >= nt) {               // past this tile's last key tile (or tile unused): release V_j
                mbar_arrive(smem_u32(&bars->v_empty[cv % NV]));
                continue;
            }
            ok = wait_bar(smem_u32(&bars->p_full[t]), npv & 1, abort, kErrWaitMma + 6 + t);
            if (ok && j == 0 && units > 0)
                ok = wait_bar(smem_u32(&bars->o_empty[t]), (units - 1) & 1, abort, kErrWaitMma + 8 + t);
            if (!ok)
                break;
            // queue order: P_t V_j goes after S_t(j+1) when the unit has one.
            // With both Q tiles sharing one S region, S is on the chain (its
            // softmax reads it, then the other tile's S may use the region)
            // and this P V has a tile of slack.  A hint only (no data hazard
            // either way): a bounded spin, then go on.  Measured: +7 % on
            // causal GQA S=4096 D=128; a loss with per-tile S regions (D=64),
            // for E4M3 and for the decode units, which keep the arrival order.
            if (L::kSharedS && KIND != kE4M3 && !kPacked && j + 1 < nt) {
                const volatile uint32_t* issued = &bars->s_issued[t];
                for (int spin = 0; spin < kOrderSpins && *issued < npv + 2; ++spin) {
                }
            }
            tc_fence_after_sync();
            const uint32_t v_lo = v_lo0 + (cv % NV) * kTileUnits;
#pragma unroll
            for (int kk = 0; kk < L::kPVSteps; ++kk) {
                const uint32_t off_v = (uint32_t)((kk * L::kKeysPerStep * L::kSwz) >> 4);
                const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
                if constexpr (kFP8)
                    mma_f8_ss(o_tmem, desc_join(p_hi, p_lo + (uint32_t)(kk * 2)), desc_join(desc_hi, v_lo + off_v),
                              idesc_o, acc);
                else
                    mma_f16_ts(o_tmem, p_tmem + kk * 8, desc_join(desc_hi, v_lo + off_v), idesc_o, acc);
            }
            if constexpr (kFP8) {
#pragma unroll
                for (int kk = 0; kk < L::kPVSteps; ++kk)
                    mma_f8_ss(l_tmem, desc_join(p_hi, p_lo + (uint32_t)(kk * 2)),
                              desc_join(p_hi, ones_lo + (uint32_t)(kk * 2)), idesc_l, (j > 0 || kk > 0) ? 1u : 0u);
            }
            mma_commit(smem_u32(&bars->pv_done[t]));
            mma_commit(smem_u32(&bars->v_empty[cv % NV]));
            if (j == nt - 1)
                mma_commit(smem_u32(&bars->o_full[t]));
            ++npv;
        }
        units += (nt > 0) ? 1u : 0u;
    }
    mma_commit(smem_u32(&bars->drain[t]));
    drain_wait(smem_u32(&bars->drain[t]), 0);
}

// tm_o: O as [B][Sq][Hq][D] with the caller's strides, box {kOSwz bytes of a
// row, 1 head, 32 rows, 1 batch}; unused in packed mode.
template <int D, int KIND, bool kPacked, int QT = 2>
__global__ void __launch_bounds__(Roles<QT>::kThreads, Roles<QT>::kCtasPerSm)
sdpa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o, const Params p)
{
    using L = Layout<D, KIND, QT>;
    using R = Roles<QT>;
    constexpr bool kFP8 = (KIND == kE4M3);
    constexpr bool kOutBF16 = (KIND != kFP16);         // E4M3 inputs give a bf16 output
    constexpr int NK = L::kStagesK;
    constexpr int NV = L::kStagesV;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    auto* bars = reinterpret_cast<Barriers<NK, NV>*>(smem + L::kOffBar);
    volatile int* abort = &bars->abort;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    const uint32_t sQ = smem_u32(smem + L::kOffQ);
    const uint32_t sK = smem_u32(smem + L::kOffK);
    const uint32_t sV = smem_u32(smem + L::kOffV);
    const uint32_t sP = smem_u32(smem + L::kOffP);     // E4M3 only
    const uint32_t sO = smem_u32(smem + L::kOffO);     // output staging

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            mbar_init(smem_u32(&bars->q_full[t]), 1);
            mbar_init(smem_u32(&bars->q_empty[t]), 1);
            mbar_init(smem_u32(&bars->s_full[t]), 1);
            mbar_init(smem_u32(&bars->p_full[t]), 128);
            mbar_init(smem_u32(&bars->o_full[t]), 1);
            mbar_init(smem_u32(&bars->o_empty[t]), 128);
            mbar_init(smem_u32(&bars->pv_done[t]), 1);
        }
        for (int s = 0; s < NK; ++s) {
            mbar_init(smem_u32(&bars->k_full[s]), 1);
            mbar_init(smem_u32(&bars->k_empty[s]), 1);          // released by the S issuer
        }
        for (int s = 0; s < NV; ++s) {
            mbar_init(smem_u32(&bars->v_full[s]), 1);
            mbar_init(smem_u32(&bars->v_empty[s]), QT);         // released by every P V issuer
        }
        mbar_init(smem_u32(&bars->s_free[0]), 128);
        mbar_init(smem_u32(&bars->s_free[1]), 128);
        for (int i = 0; i < 3; ++i)
            mbar_init(smem_u32(&bars->drain[i]), 1);
        bars->abort = 0;
        bars->s_issued[0] = bars->s_issued[1] = 0;
        fence_mbar_init();
    }
    if (warp == R::kProducerWarp && lane == 0) {
        tma_prefetch_map(&tm_q);
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_v);
        if constexpr (!kPacked)
            tma_prefetch_map(&tm_o);
    }
    if (warp == R::kMmaWarp) {
        tmem_alloc(smem_u32(&bars->tmem_base), L::kTmemCols);
        tmem_relinquish();
    }
    if constexpr (kFP8) {
        uint32_t* ones = reinterpret_cast<uint32_t*>(smem + L::kOffOnes);
        for (int i = threadIdx.x; i < L::kOnesBytes / 4; i += R::kThreads)
            ones[i] = 0x38383838u;
        fence_proxy_async_smem();                      // read by tcgen05.mma
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    // Everything above touches only this CTA's shared memory, TMEM and the
    // kernel's parameters, so with a programmatic dependent launch it runs
    // while the previous kernel in the stream finishes.  Global memory (inputs
    // that kernel may still be writing, outputs it may still be reading) only
    // after it has completed; then the next launch may be scheduled.
    grid_dependency_wait();
    grid_launch_dependents();

    if (warp >= R::kProducerWarp) {
      regs_release<R::kRegsProducer>();
      if (warp == R::kProducerWarp) {
        // =========================== TMA producer ===========================
        if (lane == 0) {
            uint32_t nk = 0, nv = 0;             // K / V tiles issued (ring position)
            uint32_t nq[2] = {0, 0};             // Q tiles issued per slot
            bool ok = true;
            auto load_q = [&](const Unit& w, int t) -> bool {
                if (nq[t] > 0 && !wait_bar(smem_u32(&bars->q_empty[t]), (nq[t] - 1) & 1, abort, kErrWaitLoad + 1 + t))
                    return false;
                mbar_arrive_expect_tx(smem_u32(&bars->q_full[t]), L::kTileBytes);
                // packed: the tensor map's box is {chunk, G heads, 128 / G positions},
                // so one copy brings rows s * G + h of the KV head's query heads
                const int r0 = w.pair * R::kUnitRows + t * kBlockM;
                const int h = kPacked ? w.hkv * p.group : w.hq;
                const int s0 = kPacked ? r0 / p.group : r0;
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_4d(sQ + t * L::kTileBytes + c * L::kChunkBytes, &tm_q, smem_u32(&bars->q_full[t]),
                                c * (L::kSwz / L::kEsize), h, s0, w.b);
                ++nq[t];
                return true;
            };
            auto load_k = [&](const Unit& w, int j) -> bool {
                const uint32_t s = nk % NK;
                if (nk >= NK && !wait_bar(smem_u32(&bars->k_empty[s]), ((nk / NK) & 1) ^ 1, abort, kErrWaitLoad + 3))
                    return false;
#ifdef SDPA_WAIT_TEST
                if ((int)nk == g_test_withhold_k) {        // test build: this K copy is never issued
                    ++nk;
                    return true;
                }
#endif
                mbar_arrive_expect_tx(smem_u32(&bars->k_full[s]), L::kTileBytes);
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_4d(sK + s * L::kTileBytes + c * L::kChunkBytes, &tm_k, smem_u32(&bars->k_full[s]),
                                c * (L::kSwz / L::kEsize), w.hkv, (w.kv0 + j) * kBlockN, w.b);
                ++nk;
                return true;
            };
            auto load_v = [&](const Unit& w, int j) -> bool {
                const uint32_t s = nv % NV;
                if (nv >= NV && !wait_bar(smem_u32(&bars->v_empty[s]), ((nv / NV) & 1) ^ 1, abort, kErrWaitLoad + 4))
                    return false;
                mbar_arrive_expect_tx(smem_u32(&bars->v_full[s]), L::kTileBytes);
                for (int c = 0; c < L::kChunks; ++c)
                    tma_load_4d(sV + s * L::kTileBytes + c * L::kChunkBytes, &tm_v, smem_u32(&bars->v_full[s]),
                                c * (L::kSwz / L::kEsize), w.hkv, (w.kv0 + j) * kBlockN, w.b);
                ++nv;
                return true;
            };
            for (int r = 0; ok; ++r) {
                const int u = unit_of_round(p, r);
                if (u == -2)
                    break;
                if (u < 0)
                    continue;
                const Unit w = decode_unit<kPacked, QT>(p, u);
                const int n = w.n;
                ok = load_q(w, 0) && load_k(w, 0) && (w.n_kv[1] == 0 || load_q(w, 1)) && load_v(w, 0);
                for (int j = 1; ok && j < n; ++j)
                    ok = load_k(w, j) && load_v(w, j);
            }
            {
                // never leave the CTA with copies in flight: wait (bounded)
                // for the last use of every slot -- at once in a normal run,
                // where the consumers have waited for them; after an abort,
                // for the copies still landing
                for (int t = 0; t < 2; ++t)
                    if (nq[t] > 0)
                        drain_wait(smem_u32(&bars->q_full[t]), (nq[t] - 1) & 1);
                for (uint32_t i = (nk > NK ? nk - NK : 0); i < nk; ++i)
                    drain_wait(smem_u32(&bars->k_full[i % NK]), (i / NK) & 1);
                for (uint32_t i = (nv > NV ? nv - NV : 0); i < nv; ++i)
                    drain_wait(smem_u32(&bars->v_full[i % NV]), (i / NV) & 1);
            }
        }
      } else if (warp == R::kSMmaWarp) {
        // ============================= S issuer =============================
        if (lane == 0)
            mma_issue_s<D, KIND, kPacked, NK, NV, QT>(p, bars, abort, tmem, sQ, sK);
      } else if (warp >= R::kMmaWarp && warp < R::kMmaWarp + QT) {
        // =========================== P V issuers ============================
        if (lane == 0) {
            mma_issue_pv<D, KIND, kPacked, NK, NV, QT>(p, bars, abort, tmem, sV, sP, smem_u32(smem + L::kOffOnes),
                                                  warp - R::kMmaWarp);
        }
      }
    } else {
        regs_acquire<R::kRegsSoftmax>();
        // ========================= softmax warpgroups =======================
        const int t = warp >> 2;                           // Q tile of this warpgroup
        const int quarter = warp & 3;                      // TMEM lanes 32*quarter ..
        const int row = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const uint32_t s_tmem = tmem + lane_addr + L::tmem_s(t);
        const uint32_t o_tmem = tmem + lane_addr + L::tmem_o(t);
        const float c = p.scale_log2;
        uint32_t cs = 0;                                   // S tiles consumed
        uint32_t np = 0;                                   // P tiles handed to the MMA
        uint32_t units = 0;
        bool ok = true;
        const uint32_t p_row = sP + t * L::kPTileBytes + row * 128;   // E4M3: this row of P_t
        const uint32_t l_tmem = tmem + lane_addr + L::tmem_l(t);      // E4M3: row sum of P_t
        const uint32_t p_tmem = tmem + lane_addr + L::tmem_p(t);      // 16-bit: P_t
        // O_t *= alpha in TMEM (the running max grew past the threshold)
        auto rescale_o = [&](float alpha) {
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
                uint32_t o[32];
                tmem_ld32_wait(o_tmem + cc * 32, o);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                tmem_st32(o_tmem + cc * 32, o);
            }
        };
        for (int r = 0; ok; ++r) {
            const int u = unit_of_round(p, r);
            if (u == -2)
                break;
            if (u < 0)
                continue;
            const Unit w = decode_unit<kPacked, QT>(p, u);
            const int n = w.kv(t);
            if (n == 0)
                continue;                                  // this Q tile has no rows in the unit
            // this thread's row: query position q_idx of head hq (packed:
            // row r of the KV head's stacked heads, r = q_idx * G + head)
            const int r_all = w.pair * R::kUnitRows + t * kBlockM + row;
            const int q_idx = kPacked ? r_all / p.group : r_all;
            const int hq = kPacked ? w.hkv * p.group + r_all % p.group : w.hq;
            int limit = p.Skv - 1;                         // last key this row sees
            if (p.causal && q_idx < limit)
                limit = q_idx;
            float m = -INFINITY;                           // running max of S*c
            float l = 0.f;                                 // running sum of exp2(S*c - m) (16-bit kinds)
            for (int j = 0; j < n; ++j) {
                ok = __all_sync(0xffffffffu,
                                wait_bar(smem_u32(&bars->s_full[t]), cs & 1, abort, kErrWaitSoftmax + 1 + t));
                if (!ok)
                    break;
                ++cs;
                tc_fence_after_sync();
                uint32_t r[128];
                tmem_ld128_wait(s_tmem, s_tmem + 32, s_tmem + 64, s_tmem + 96, r);
                // the S region is free for the next S as soon as it is read
                tc_fence_before_sync();
                mbar_arrive(smem_u32(&bars->s_free[t]));
                const int k0 = (w.kv0 + j) * kBlockN;
                if (k0 + kBlockN - 1 > limit) {
#pragma unroll
                    for (int i = 0; i < 128; ++i)
                        if (k0 + i > limit)
                            r[i] = 0xff800000u;            // -inf
                }
                // row max: four chains of three-operand max
                float mx0 = __uint_as_float(r[0]), mx1 = __uint_as_float(r[1]);
                float mx2 = __uint_as_float(r[2]), mx3 = __uint_as_float(r[3]);
#pragma unroll
                for (int i = 4; i < 124; i += 8) {              // elements 4..123
                    mx0 = fmax3(mx0, __uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                    mx1 = fmax3(mx1, __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
                    mx2 = fmax3(mx2, __uint_as_float(r[i + 4]), __uint_as_float(r[i + 5]));
                    mx3 = fmax3(mx3, __uint_as_float(r[i + 6]), __uint_as_float(r[i + 7]));
                }
                mx0 = fmax3(mx0, __uint_as_float(r[124]), __uint_as_float(r[125]));
                mx1 = fmax3(mx1, __uint_as_float(r[126]), __uint_as_float(r[127]));
                const float m_tile = fmax3(fmaxf(mx0, mx1), mx2, mx3) * c;
                float alpha = 1.f;
                bool rescale = false;
                if (j == 0) {
                    m = m_tile;
                } else if (m_tile > m + (kFP8 ? kRescaleThresholdFP8 : kRescaleThreshold)) {
                    alpha = ex2_approx(m - m_tile);
                    m = m_tile;
                    rescale = true;
                }
                const uint64_t c2 = f32x2(c, c);
                if constexpr (!kFP8) {
                    // P = exp2(S*c - m) as 16-bit: packed FMA for the
                    // argument, packed adds for the fp32 row sum
                    const uint64_t nm2 = f32x2(-m, -m);
                    uint64_t acc0 = f32x2(0.f, 0.f), acc1 = acc0;
                    uint32_t pk[2][32];
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        float x0, x1;
                        f32x2_split(fma_f32x2(f32x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), c2, nm2),
                                    x0, x1);
                        const float p0 = ex2_approx(x0);
                        const float p1 = ex2_approx(x1);
                        if (i & 1)
                            acc1 = add_f32x2(acc1, f32x2(p0, p1));
                        else
                            acc0 = add_f32x2(acc0, f32x2(p0, p1));
                        pk[i >> 5][i & 31] = pack2<kOutBF16>(p0, p1);
                    }
                    // the previous P_t V has read P_t's columns and updated O_t
                    if (np > 0)
                        ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->pv_done[t]), (np - 1) & 1, abort,
                                                              kErrWaitSoftmax + 5 + t));
                    if (!ok)
                        break;
                    ++np;
                    tc_fence_after_sync();
                    if (__any_sync(0xffffffffu, rescale))
                        rescale_o(alpha);
                    tmem_st32(p_tmem, pk[0]);
                    tmem_st32(p_tmem + 32, pk[1]);
                    tmem_st_wait();
                    tc_fence_before_sync();
                    mbar_arrive(smem_u32(&bars->p_full[t]));
                    float sa, sb;
                    f32x2_split(add_f32x2(acc0, acc1), sa, sb);
                    l = l * alpha + (sa + sb);
                } else {
                    // P8 = E4M3(exp2(S*c - m) * 56), four keys per 32-bit word
                    const float bias = m - kLog2P8Scale;
                    const uint64_t nb2 = f32x2(-bias, -bias);
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int e = 4 * i;
                        float x0, x1, x2, x3;
                        f32x2_split(fma_f32x2(f32x2(__uint_as_float(r[e]), __uint_as_float(r[e + 1])), c2, nb2), x0, x1);
                        f32x2_split(fma_f32x2(f32x2(__uint_as_float(r[e + 2]), __uint_as_float(r[e + 3])), c2, nb2), x2,
                                    x3);
                        const uint32_t lo = f32x2_to_e4m3x2(ex2_approx(x0), ex2_approx(x1));
                        const uint32_t hi = f32x2_to_e4m3x2(ex2_approx(x2), ex2_approx(x3));
                        pk[i] = lo | (hi << 16);
                    }
                    // the previous P_t V has read the P_t buffer and updated O_t
                    if (np > 0)
                        ok = __all_sync(0xffffffffu, wait_bar(smem_u32(&bars->pv_done[t]), (np - 1) & 1, abort,
                                                              kErrWaitSoftmax + 5 + t));
                    if (!ok)
                        break;
                    ++np;
                    tc_fence_after_sync();
                    if (__any_sync(0xffffffffu, rescale)) {
                        rescale_o(alpha);
                        tmem_st1(l_tmem, __float_as_uint(__uint_as_float(tmem_ld1_wait(l_tmem)) * alpha));
                    }
                    // this row's 128 keys: one 128-byte row of the K-major P
                    // tile, 16-byte chunk c at position c ^ (row & 7)
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc)
                        st_shared_v4(p_row + (uint32_t)((cc ^ (row & 7)) << 4), pk[4 * cc], pk[4 * cc + 1],
                                     pk[4 * cc + 2], pk[4 * cc + 3]);
                    fence_proxy_async_smem();
                    tmem_st_wait();
                    tc_fence_before_sync();
                    mbar_arrive(smem_u32(&bars->p_full[t]));
                }
            }
            if (!ok)
                break;
            // ---- epilogue: O_t / l -> 16-bit -> HBM -------------------------
            ok = __all_sync(0xffffffffu,
                            wait_bar(smem_u32(&bars->o_full[t]), units & 1, abort, kErrWaitSoftmax + 3 + t));
            if (!ok)
                break;
            tc_fence_after_sync();
            uint32_t o[D];
            if constexpr (D == 128) {
                tmem_ld128_wait(o_tmem, o_tmem + 32, o_tmem + 64, o_tmem + 96, o);
            } else {
#pragma unroll
                for (int cc = 0; cc < D / 32; ++cc)
                    tmem_ld32_wait(o_tmem + 32 * cc, *reinterpret_cast<uint32_t(*)[32]>(&o[32 * cc]));
            }
            if constexpr (kFP8)
                l = __uint_as_float(tmem_ld1_wait(l_tmem));   // sum of the E4M3 P values (tensor core, fp32)
            tc_fence_before_sync();
            mbar_arrive(smem_u32(&bars->o_empty[t]));
            const float inv_l = p.out_scale / l;
            const int64_t row_id = ((int64_t)w.b * p.Hq + hq) * p.Sq + q_idx;
            if (q_idx < p.Sq && (p.lse || (kPacked && p.part_o))) {
                // log sum_j exp(s_j) = ln 2 * (m + log2 l): m is the max of
                // s * log2(e) the weights were taken against, l their sum
                // (E4M3: of the weights times 56)
                const float lse = (m + (kFP8 ? log2f(l) - kLog2P8Scale : log2f(l))) * kLn2;
                if (kPacked && p.part_o)
                    p.part_lse[row_id * p.n_splits + w.split] = lse;
                else
                    p.lse[row_id] = lse;
            }
            if constexpr (kPacked) {
                if (q_idx < p.Sq) {
                    if (p.part_o) {
                        // one split of the key range: O / l in fp32, merged later
                        float4* dst = reinterpret_cast<float4*>(p.part_o + (row_id * p.n_splits + w.split) * D);
#pragma unroll
                        for (int v = 0; v < D / 4; ++v)
                            dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv_l, __uint_as_float(o[4 * v + 1]) * inv_l,
                                                 __uint_as_float(o[4 * v + 2]) * inv_l,
                                                 __uint_as_float(o[4 * v + 3]) * inv_l);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.O) +
                                                              ((int64_t)w.b * p.o_sb + (int64_t)q_idx * p.o_ss +
                                                               (int64_t)hq * p.o_sh) * 2);
#pragma unroll
                        for (int v = 0; v < D / 8; ++v)
                            dst[v] = make_uint4(
                                pack2<kOutBF16>(__uint_as_float(o[8 * v + 0]) * inv_l, __uint_as_float(o[8 * v + 1]) * inv_l),
                                pack2<kOutBF16>(__uint_as_float(o[8 * v + 2]) * inv_l, __uint_as_float(o[8 * v + 3]) * inv_l),
                                pack2<kOutBF16>(__uint_as_float(o[8 * v + 4]) * inv_l, __uint_as_float(o[8 * v + 5]) * inv_l),
                                pack2<kOutBF16>(__uint_as_float(o[8 * v + 6]) * inv_l, __uint_as_float(o[8 * v + 7]) * inv_l));
                    }
                }
            } else {
                // O / l -> 16-bit rows of this warp in its staging area (row
                // = lane, 16-byte units swizzled as the TMA store reads them:
                // unit u of row r at u ^ (r & 7), or u ^ ((r >> 1) & 3) for
                // 64-byte rows), then one TMA store per pass.  Rows past Sq
                // are clipped by the store.
                const uint32_t stage = sO + (uint32_t)warp * L::kOWarpBytes;
                const int q_warp = w.pair * R::kUnitRows + t * kBlockM + quarter * 32;   // first row of the warp
                constexpr int kUnits = L::kOSwz / 16;
                const uint32_t swz = (L::kOSwz == 128) ? (uint32_t)(lane & 7) : (uint32_t)((lane >> 1) & 3);
#pragma unroll
                for (int c = 0; c < L::kOPasses; ++c) {
                    // the previous store from this staging area has read it
                    if (lane == 0)
                        bulk_wait_group_read0();
                    __syncwarp();
#pragma unroll
                    for (int u = 0; u < kUnits; ++u) {
                        const int e = c * (L::kOSwz / 2) + 8 * u;      // first of the unit's 8 elements
                        st_shared_v4(stage + (uint32_t)(lane * L::kOSwz) + (((uint32_t)u ^ swz) << 4),
                                     pack2<kOutBF16>(__uint_as_float(o[e + 0]) * inv_l, __uint_as_float(o[e + 1]) * inv_l),
                                     pack2<kOutBF16>(__uint_as_float(o[e + 2]) * inv_l, __uint_as_float(o[e + 3]) * inv_l),
                                     pack2<kOutBF16>(__uint_as_float(o[e + 4]) * inv_l, __uint_as_float(o[e + 5]) * inv_l),
                                     pack2<kOutBF16>(__uint_as_float(o[e + 6]) * inv_l, __uint_as_float(o[e + 7]) * inv_l));
                    }
                    fence_proxy_async_smem();                  // visible to the TMA engine
                    __syncwarp();
                    if (lane == 0 && q_warp < p.Sq) {
                        tma_store_4d(&tm_o, stage, c * (L::kOSwz / 2), hq, q_warp, w.b);
                        bulk_commit_group();
                    }
                }
            }
            ++units;
        }
        // every output store has completed before the CTA exits
        if (!kPacked && lane == 0)
            bulk_wait_group0();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == R::kMmaWarp) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

// Merges the key-range splits of a packed (decode) pass.  Split k of a row
// holds its normalised output O_k = sum_{j in k} w_j V_j / l_k and lse_k =
// log l_k (with the max folded in); over all splits
//     LSE = log sum_k exp(lse_k),   O = sum_k exp(lse_k - LSE) O_k,
// the same softmax over the whole key range.  One warp per row (b, hq, s);
// each lane merges D / 32 consecutive columns.
template <int D, bool kOutBF16>
__global__ void __launch_bounds__(128) sdpa_combine_kernel(const Params p)
{
    constexpr int kCols = D / 32;
    const int64_t row = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= (int64_t)p.B * p.Hq * p.Sq)
        return;
    const int S = p.n_splits;
    const float* lse = p.part_lse + row * S;
    float mx = -INFINITY;
    for (int k = 0; k < S; ++k)
        mx = fmaxf(mx, lse[k]);
    float den = 0.f;
    float acc[kCols];
#pragma unroll
    for (int c = 0; c < kCols; ++c)
        acc[c] = 0.f;
    for (int k = 0; k < S; ++k) {
        const float w = expf(lse[k] - mx);
        den += w;
        const float* o = p.part_o + (row * S + k) * D + lane * kCols;
#pragma unroll
        for (int c = 0; c < kCols; ++c)
            acc[c] += w * o[c];
    }
    const float inv = 1.f / den;
    const int q = (int)(row % p.Sq);
    const int64_t bh = row / p.Sq;
    const int hq = (int)(bh % p.Hq);
    const int b = (int)(bh / p.Hq);
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.O) + (int64_t)b * p.o_sb + (int64_t)q * p.o_ss +
                    (int64_t)hq * p.o_sh + lane * kCols;
    if constexpr (kCols % 2 == 0) {
#pragma unroll
        for (int c = 0; c < kCols; c += 2)
            *reinterpret_cast<uint32_t*>(dst + c) = pack2<kOutBF16>(acc[c] * inv, acc[c + 1] * inv);
    } else {
#pragma unroll
        for (int c = 0; c < kCols; ++c)
            dst[c] = (uint16_t)(pack2<kOutBF16>(acc[c] * inv, 0.f) & 0xffffu);
    }
    if (p.lse && lane == 0)
        p.lse[row] = mx + logf(den);
}

}  // namespace sdpa
