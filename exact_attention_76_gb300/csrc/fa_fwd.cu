// Forward attention kernel for sm_103a (bf16 and e4m3 inputs).
//
// What it computes ("FLASH-ATTN", FlashAttention-2 > FlashAttention-2): for a
// block of query rows, a loop over key/value blocks keeps a running row max m,
// a running row sum l of exp(S - m) and an UNSCALED output accumulator
// O~ = sum_j exp(S_j - m) V_j; O = diag(l)^-1 O~ and L = m + log(l) are formed
// once after the loop.  Fully masked blocks of a causal row block are never
// visited and only the blocks that cross the diagonal apply the element mask
// (same section).  Query blocks are independent thread blocks (> Parallelism).
//
// How it maps to the SM (one CTA = 256 query rows of one (batch, head)):
//  * warps 0-3 and 4-7: two softmax warpgroups, one per 128-row query tile;
//    thread r of a warpgroup owns row r (TMEM lane r);
//  * warp 8: TMA producer -- the two Q tiles once, then K_j and V_j (128 keys
//    each) into a ring of shared-memory slots guarded by full/empty mbarriers
//    (the producer/consumer split of "FLASH-ATTN", FlashAttention-3 >
//    Producer-Consumer asynchrony);
//  * warp 9: allocates TMEM and, from one thread, issues every tcgen05.mma:
//    S_t = Q_t K_j^T (both operands in shared memory) and O_t += P_t V_j with
//    P_t read from TMEM.
//
// Per query tile t the tensor core computes S_t(j) with N = 128 keys; the
// softmax warpgroup reads S_t(j) into registers and writes P_t(j) into the
// first columns of S_t's own TMEM space; the MMA thread then issues
// O_t += P_t(j) V_j and, at once, S_t(j+1) into the same columns.  The
// tcgen05.mma operations of one thread execute in issue order, so S_t(j+1)
// overwrites P_t(j) only after PV_t(j) has read it, with no wait in between.
// The two tiles alternate on the tensor core (PV_0, S_0, PV_1, S_1, ...), so
// one warpgroup's softmax overlaps the other tile's two products (the
// ping-pong of two consumer warpgroups, "FLASH-ATTN", FlashAttention-3).  A
// completed S_t(j) also means that PV_t(j-1), issued before it, is complete,
// so the warpgroup may rescale O_t right after reading S_t(j).  In bf16 P is
// handed over in two 64-key halves: PV over the first half runs while the
// warpgroup exponentiates the second.
//
// FP8 at d = 128 splits S_t into two 64-key halves with P over the second, so
// that the next block's first half is computed while the softmax runs (see
// FwdCfg::kSplitS).
//
// At d = 64 (O takes half the columns) P_t has TMEM columns of its own, and
// the order changes: the warpgroup signals s_free as soon as S_t(j) is in its
// registers, the MMA thread then issues S_t(j+1) at once, and PV_t(j) after
// the hand-over of P_t(j); the warpgroup waits for PV_t(j-1) to complete
// (o_done) only before its first TMEM write of block j.  The next block's S
// is then ready when the softmax of this one ends.
//
// Softmax works in the log2 domain: x = S * (scale * log2 e) with one FMA, then
// ex2.  The reference maximum m_used is raised only when a block's maximum
// exceeds it by more than TAU (8 for bf16, i.e. values up to 2^8 before a
// rescale; 4 for e4m3, whose P * 2^4 must stay below 448); raising it
// rescales l and the warpgroup's own O row in TMEM.  Any TAU gives the same
// exact result.  Each exponential is packed into its P word as soon as it is
// computed; the e4m3 factor 2^4 is folded into the exponent.
//
// TMEM columns: S_0 [0,128), S_1 [128,256) (at d = 128, P_t in the first 64
// columns of S_t for bf16, columns 64-95 for e4m3), O_0 [256,256+D),
// O_1 [256+D,256+2D), and at d = 64 P_0 [384,448), P_1 [448,512).
// Q stays in shared memory: an M = 128, N = 128 product with both operands in
// shared memory uses the full shared-memory operand bandwidth, not more
// (measured: 64 cycles per K = 16 step, the tensor core's own rate); with
// 64-key blocks the N = 64 products of S took 48-50 cycles for half the work.
#include <cuda_bf16.h>

#include <algorithm>

#include "fa_common.cuh"
#include "fa_host.h"

namespace fa {

namespace {

__device__ uint32_t g_err_fwd;

constexpr int kThreads = 320;
constexpr int kBM = 128;  // query rows per tile (one TMEM lane each)
constexpr int kHalf = 64;  // keys per half block (one exp2_pack_row call)

__device__ __forceinline__ void issue_mma(bool fp8, uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if (fp8) mma_f8_ss(d, a, b, idesc, acc);
  else mma_bf16_ss(d, a, b, idesc, acc);
}
__device__ __forceinline__ void issue_mma_ts(bool fp8, uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                             uint32_t acc) {
  if (fp8) mma_f8_ts(d, a, b, idesc, acc);
  else mma_bf16_ts(d, a, b, idesc, acc);
}

// P for 64 keys of one row: p_i = 2^(s_i * c - m), packed into the words
// written to TMEM (bf16 pairs, or four e4m3); returns the sum of the p_i.  The
// scores s are left unchanged.  EMU of the 16 groups of four use the
// polynomial exp2 (spread evenly), the rest ex2.approx.  With PMUL the e4m3
// words hold p_i * pmul (the block-quantised V's relative scale).
template <bool FP8, int EMU, int DEG, bool PMUL = false>
__device__ __forceinline__ float exp2_pack_row(const float (&s)[kHalf], float c, float m,
                                               uint32_t (&pw)[FP8 ? kHalf / 4 : kHalf / 2], float pmul = 1.0f) {
  const float2 c2 = make_float2(c, c);
  const float2 nm2 = make_float2(-m, -m);
  float2 part0 = make_float2(0.f, 0.f), part1 = make_float2(0.f, 0.f);
#pragma unroll
  for (int i = 0; i < kHalf; i += 4) {
    const int g = i / 4;
    const float2 x0 = __ffma2_rn(make_float2(s[i], s[i + 1]), c2, nm2);
    const float2 x1 = __ffma2_rn(make_float2(s[i + 2], s[i + 3]), c2, nm2);
    float2 y0, y1;
    if (((g + 1) * EMU) / (kHalf / 4) != (g * EMU) / (kHalf / 4)) {
      y0 = exp2_poly2<DEG>(x0);
      y1 = exp2_poly2<DEG>(x1);
    } else {
      y0 = make_float2(ex2_approx(x0.x), ex2_approx(x0.y));
      y1 = make_float2(ex2_approx(x1.x), ex2_approx(x1.y));
    }
    part0 = __fadd2_rn(part0, y0);
    part1 = __fadd2_rn(part1, y1);
    if constexpr (FP8 && PMUL) {  // the operand carries a factor, the sum does not
      const float2 z0 = __fmul2_rn(y0, make_float2(pmul, pmul));
      const float2 z1 = __fmul2_rn(y1, make_float2(pmul, pmul));
      pw[g] = pack_e4m3x4(z0.x, z0.y, z1.x, z1.y);
    } else if constexpr (FP8) {
      pw[g] = pack_e4m3x4(y0.x, y0.y, y1.x, y1.y);
    } else {
      pw[2 * g] = pack_bf16x2(y0.x, y0.y);
      pw[2 * g + 1] = pack_bf16x2(y1.x, y1.y);
    }
  }
  return (part0.x + part0.y) + (part1.x + part1.y);
}

// Block index -> (query head, query block).  Query heads are taken in groups
// whose keys and values stay in L2 together while every query block of the
// group streams them; within a group, under a causal mask, the query blocks
// that see the most keys (the last) come first.  A partial group (the
// remainder of BH / group) goes first, so that the launch ends on the light
// blocks of a full group.
__device__ __forceinline__ void fwd_item(int item, int BH, int n_qblk, int group, int causal, int& bh, int& qb) {
  const int rem = BH % group;
  int g_heads, base_item, base_head;
  if (item < rem * n_qblk) {
    g_heads = rem;
    base_item = 0;
    base_head = 0;
  } else {
    const int g = (item - rem * n_qblk) / (group * n_qblk);
    g_heads = group;
    base_item = rem * n_qblk + g * group * n_qblk;
    base_head = rem + g * group;
  }
  const int r = item - base_item;
  const int step = r / g_heads;
  qb = causal ? n_qblk - 1 - step : step;
  bh = base_head + (r - step * g_heads);
}

constexpr int kBN = 128;  // keys per key/value block

template <int D, bool FP8>
struct FwdCfg {
  static constexpr int kElemBytes = FP8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElemBytes;
  // Swizzle width of Q, K and V in shared memory: 128 bytes, or 64 when a row
  // is 64 bytes (e4m3 at d = 64).
  static constexpr int kSwz = kRowBytes >= 128 ? 128 : 64;
  static constexpr int kColBlocks = kRowBytes / kSwz;     // kSwz-byte column blocks
  static constexpr int kBoxCols = kSwz / kElemBytes;
  static constexpr int kBlockBytes = 128 * kSwz;         // one 128-row column block
  static constexpr int kStepsPerBlock = kSwz / 32;       // K steps of 32 bytes per column block
  static constexpr int kTileBytes = 128 * kRowBytes;     // a Q tile or a K / V block
  // O (bf16, 128-byte swizzle) is staged in the tile's Q space: kORows rows
  // of kOStageBlocks 128-byte column blocks at a time.
  static constexpr int kOColBlocks = D * 2 / 128;
  static constexpr int kORows = kTileBytes / 128 >= 128 ? 128 : kTileBytes / 128;
  static constexpr int kOStageBytes = kORows * 128;     // one staged column block
  static constexpr int kOStageBlocks = kTileBytes / kOStageBytes;
  static constexpr int kSlotsFit = (232448 - 1024 - 1024 - 2 * kTileBytes) / kTileBytes;
  static constexpr int kSlots = kSlotsFit > 16 ? 16 : kSlotsFit;
  static constexpr int kSmemBytes = 2 * kTileBytes + kSlots * kTileBytes + 1024;
  static constexpr int kKPerMma = FP8 ? 32 : 16;
  static constexpr int kQKSteps = kRowBytes / 32;
  static constexpr int kPVSteps = kBN / kKPerMma;
  static constexpr float kTauLog2 = FP8 ? 4.0f : 8.0f;
  static constexpr float kPShiftLog2 = FP8 ? -4.0f : 0.0f;
  static constexpr int kPWordsHalf = FP8 ? 16 : 32;      // TMEM words of P per 64 keys
  // P handed to the MMA thread in two 64-key halves, so that PV over the
  // first half runs while the second half is exponentiated: measured +4 %
  // (causal) and +6 % (no mask) at bf16 d = 128, +1 % at d = 64; e4m3 (whose
  // PV half is only 128 tensor cycles) measured 1-2.5 % slower and hands P
  // over whole.
  static constexpr bool kSplitP = !FP8;
  // Exponentials on the FMA pipes ("software exp2"): groups of four, of the
  // 16 per 64 keys, taken by the polynomial exp2 of fa_common.cuh, and its
  // degree (bf16 P keeps 8 significant bits, e4m3 P 4).  Measured on GB300,
  // whose special-function unit delivers 32 exp2 per clock per SM, every
  // share only costs time: 2, 4 and 6 of 16 groups ran the FP8 forward 5, 6
  // and 12 % slower and the bf16 d = 128 one -2 to +1 %, so none is used.
  static constexpr int kEmuGroups = 0;
  static constexpr int kPolyDeg = FP8 ? 2 : 3;
  static constexpr uint32_t kIdescS = FP8 ? idesc_e4m3(128, kBN, false, false) : idesc_bf16(128, kBN, false, false);
  static constexpr uint32_t kIdescPV = FP8 ? idesc_e4m3(128, D, false, true) : idesc_bf16(128, D, false, true);
  static constexpr uint32_t kTmS = 0;     // + t * 128
  static constexpr uint32_t kTmO = 256;   // + t * D
  // At d = 64 TMEM has room for P in columns of its own (384 + t * 64), so
  // S_t(u+1) is issued as soon as the warpgroup has read S_t(u) and runs while
  // the warpgroup exponentiates (measured: +17 % on the bf16 d = 64 forward at
  // N = 8192 and 16384, +10 % in FP8, +3-8 % at N = 512 and 1024); at d = 128
  // P is written over S_t.
  static constexpr bool kEarlyS = (D == 64);
  // FP8 at d = 128 computes S_t in two 64-key halves: P_t(j) (32 columns) is
  // written over the second half's columns, so the first half of S_t(j+1) is
  // issued as soon as the warpgroup has read S_t(j)'s first half, and only the
  // second half follows PV_t(j) in issue order; the warpgroup reduces the
  // first half's maximum while the second is computed.  Measured +5-6 % in
  // FP8 (tensor-pipe active cycles per launch unchanged); bf16, whose PV is
  // twice as long, measured 8-11 % slower with the same split.
  static constexpr bool kSplitS = FP8 && D == 128;
  static constexpr uint32_t kIdescSHalf =
      FP8 ? idesc_e4m3(128, kBN / 2, false, false) : idesc_bf16(128, kBN / 2, false, false);
  static constexpr uint32_t kTmP = kEarlyS ? 384 : 0;  // + t * 64
  static_assert(!kEarlyS || kTmO + 2 * D <= kTmP, "TMEM columns");
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(kSlots >= 4, "K/V ring depth");
  static_assert(kOStageBlocks >= 1 && (kOColBlocks % kOStageBlocks == 0 || kOStageBlocks > kOColBlocks),
                "O staging");
  static_assert(kORows == 128 || kORows == 64, "O staging rows");
  static_assert(kSmemBytes <= 232448 - 1024, "shared memory budget");
};

struct FwdSmem {
  uint64_t q_full;
  uint64_t kv_full[16];
  uint64_t kv_empty[16];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t p_half[2];
  uint64_t o_done[2];
  uint64_t s_free[2];
  uint64_t s_full_b[2];
  uint64_t drain;
  uint32_t tmem_base;
  float vmax_part[2][4];
  CtaAbort abort;
};

template <int D, bool FP8, bool BS, bool WIN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                   const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
                   float* __restrict__ out_lse, const float* __restrict__ descale_q,
                   const float* __restrict__ descale_k, const float* __restrict__ descale_v, int BH, int N,
                   int causal, float scale_log2, int H, int qgroup, int window, int head_group) {
  using C = FwdCfg<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ FwdSmem sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_q = smem;                       // two Q tiles
  uint8_t* s_kv = smem + 2 * C::kTileBytes;  // ring of K/V slots

  const int warp = warp_id();
  const int n_qblk = (N + 2 * kBM - 1) / (2 * kBM);
  int bh, qb;
  fwd_item(static_cast<int>(blockIdx.x), BH, n_qblk, head_group, causal, bh, qb);
  const int bh_kv = (bh / H) * (H / qgroup) + (bh % H) / qgroup;
  const int q0 = qb * 2 * kBM;
  const int n_kv_all = (N + kBN - 1) / kBN;
  // Tile t visits key blocks j_lo[t] .. n_t[t] - 1 (len[t] of them); tile 0's
  // range starts first and the two ranges cover j_begin .. n_max - 1.
  int n_t[2], j_lo[2], len[2];
  for (int t = 0; t < 2; ++t) {
    const int row0 = q0 + t * kBM;
    if (row0 >= N) {
      n_t[t] = 0;
      j_lo[t] = 0;
    } else {
      n_t[t] = causal ? min(n_kv_all, (row0 + kBM - 1) / kBN + 1) : n_kv_all;
      j_lo[t] = WIN ? max(0, row0 - window + 1) / kBN : 0;
    }
    len[t] = n_t[t] - j_lo[t];
  }
  const int j_begin = j_lo[0];
  const int n_max = max(n_t[0], n_t[1]);

  if (threadIdx.x == 0) {
    // A wait of an earlier CTA ran out: this CTA stops after its set-up; the
    // load's latency overlaps the set-up.
    const uint32_t err0 = *reinterpret_cast<volatile uint32_t*>(&g_err_fwd);
    mbar_init(&sh.q_full, 1);
    for (int s = 0; s < C::kSlots; ++s) {
      mbar_init(&sh.kv_full[s], 1);
      mbar_init(&sh.kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&sh.s_full[t], 1);
      mbar_init(&sh.p_full[t], kBM);
      mbar_init(&sh.p_half[t], kBM);
      mbar_init(&sh.o_done[t], 1);
      mbar_init(&sh.s_free[t], kBM);
      mbar_init(&sh.s_full_b[t], 1);
    }
    mbar_init(&sh.drain, 1);
    fence_barrier_init();
    sh.abort.flag = (err0 & FA_DEVERR_TIMEOUT) ? 1 : 0;
  }
  if (warp == 9) tmem_alloc(&sh.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  if (sh.abort.flag) {
    if (warp == 9) tmem_dealloc(tmem, 512);
    return;
  }
  // Set-up done: the next kernel may start launching; inputs are read only
  // after the kernels before this one have completed.
  pdl_launch_dependents();
  pdl_wait_prior();

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (elect_one()) {
      tma_prefetch_desc(&map_q);
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      mbar_arrive_expect_tx(&sh.q_full, 2 * C::kTileBytes);
      for (int t = 0; t < 2; ++t)
        for (int cb = 0; cb < C::kColBlocks; ++cb)
          tma_load_3d(s_q + t * C::kTileBytes + cb * C::kBlockBytes, &map_q, cb * C::kBoxCols, q0 + t * kBM, bh,
                      &sh.q_full);
      int issued = 0;
      for (int j = j_begin; j < n_max && !sh.abort.flag; ++j) {
        for (int kv = 0; kv < 2; ++kv) {  // K_j then V_j
          const int slot = issued % C::kSlots;
          const int round = issued / C::kSlots;
          if (round > 0 && !mbar_wait<true>(&sh.kv_empty[slot], (round - 1) & 1, &sh.abort, &g_err_fwd)) break;
          mbar_arrive_expect_tx(&sh.kv_full[slot], C::kTileBytes);
          const CUtensorMap* m = kv == 0 ? &map_k : &map_v;
          for (int cb = 0; cb < C::kColBlocks; ++cb)
            tma_load_3d(s_kv + slot * C::kTileBytes + cb * C::kBlockBytes, m, cb * C::kBoxCols, j * kBN, bh_kv,
                        &sh.kv_full[slot]);
          ++issued;
        }
      }
      if (sh.abort.flag) {
        mbar_wait_drain(&sh.q_full, 0, &g_err_fwd);
        for (int s = 0; s < C::kSlots && s < issued; ++s) {
          const int last = s + ((issued - 1 - s) / C::kSlots) * C::kSlots;
          mbar_wait_drain(&sh.kv_full[s], (last / C::kSlots) & 1, &g_err_fwd);
        }
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one() && n_max > 0) {
      const uint64_t q_desc = sdesc_sw(smem_u32(s_q), 16, 8 * C::kSwz, C::kSwz);               // K-major Q
      const uint64_t k_desc = sdesc_sw(smem_u32(s_kv), 16, 8 * C::kSwz, C::kSwz);              // K-major K
      const uint64_t v_desc = sdesc_sw(smem_u32(s_kv), C::kBlockBytes, 8 * C::kSwz, C::kSwz);  // MN-major V
      auto issue_s = [&](int t, int slot) {
        const uint64_t a0 = sdesc_advance(q_desc, t * C::kTileBytes);
        const uint64_t b0 = sdesc_advance(k_desc, slot * C::kTileBytes);
#pragma unroll
        for (int kk = 0; kk < C::kQKSteps; ++kk) {
          const uint32_t off = (kk / C::kStepsPerBlock) * C::kBlockBytes + (kk % C::kStepsPerBlock) * 32;
          issue_mma(FP8, tmem + C::kTmS + t * kBN, sdesc_advance(a0, off), sdesc_advance(b0, off), C::kIdescS,
                    kk > 0);
        }
        tc_commit(&sh.s_full[t]);
      };
      // Half h of S_t (keys 64 h .. 64 h + 63 of the block) into S_t's columns
      // 64 h .. 64 h + 63; completion on s_full (h = 0) or s_full_b (h = 1).
      auto issue_s_half = [&](int t, int slot, int h) {
        const uint64_t a0 = sdesc_advance(q_desc, t * C::kTileBytes);
        const uint64_t b0 = sdesc_advance(k_desc, slot * C::kTileBytes + h * (kBN / 2) * C::kSwz);
#pragma unroll
        for (int kk = 0; kk < C::kQKSteps; ++kk) {
          const uint32_t off = (kk / C::kStepsPerBlock) * C::kBlockBytes + (kk % C::kStepsPerBlock) * 32;
          issue_mma(FP8, tmem + C::kTmS + t * kBN + h * (kBN / 2), sdesc_advance(a0, off), sdesc_advance(b0, off),
                    C::kIdescSHalf, kk > 0);
        }
        tc_commit(h == 0 ? &sh.s_full[t] : &sh.s_full_b[t]);
      };
      // O_t += P_t V_j over the K steps [k0, k1) of the block (P over S_t).
      auto issue_pv = [&](int t, int slot, bool acc, int k0, int k1) {
        const uint64_t b0 = sdesc_advance(v_desc, slot * C::kTileBytes);
        const uint32_t a_tm = C::kEarlyS ? tmem + C::kTmP + t * 64
                                         : tmem + C::kTmS + t * kBN + (C::kSplitS ? kBN / 2 : 0);
        const uint32_t d_tm = tmem + C::kTmO + t * D;
#pragma unroll
        for (int kk = k0; kk < k1; ++kk)
          issue_mma_ts(FP8, d_tm, a_tm + kk * 8, sdesc_advance(b0, kk * C::kKPerMma * C::kSwz), C::kIdescPV,
                       (acc || kk > 0) ? 1u : 0u);
      };
      // bf16 at d = 128 polls for P (+0.3 % causal, +1.7 % without a mask,
      // measured); elsewhere the suspending wait measured as fast or faster
      // (FP8: polling -3 %).
      auto wait_p = [&](uint64_t* bar, int u) {
        return (!FP8 && D == 128) ? mbar_wait_poll(bar, u & 1, &sh.abort, &g_err_fwd)
                                  : mbar_wait<true>(bar, u & 1, &sh.abort, &g_err_fwd);
      };
      auto wait_load = [&](int idx) {
        return mbar_wait<true>(&sh.kv_full[idx % C::kSlots], (idx / C::kSlots) & 1, &sh.abort, &g_err_fwd);
      };
      // Load index of K_j is 2 (j - j_begin), of V_j one more.
      auto k_load = [&](int j) { return 2 * (j - j_begin); };
      bool ok = mbar_wait<true>(&sh.q_full, 0, &sh.abort, &g_err_fwd) && wait_load(k_load(j_begin));
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < 2; ++t)
          if (len[t] > 0 && j_lo[t] == j_begin) {
            if constexpr (C::kSplitS) {
              issue_s_half(t, k_load(j_begin) % C::kSlots, 0);
              issue_s_half(t, k_load(j_begin) % C::kSlots, 1);
            } else {
              issue_s(t, k_load(j_begin) % C::kSlots);
            }
          }
        tc_commit(&sh.kv_empty[k_load(j_begin) % C::kSlots]);
      }
      for (int j = j_begin; ok && j < n_max; ++j) {
        const int k_idx = k_load(j + 1);  // K_(j+1)
        const int v_idx = k_load(j) + 1;  // V_j
        bool k_ready = false, v_ready = false;
        if constexpr (C::kEarlyS) {
          // S_t(u+1) as soon as the warpgroup has read S_t(u) out of its columns ...
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int v = j + 1 - j_lo[t];
            if (!ok || v < 0 || v >= len[t]) continue;
            if (v > 0) ok = mbar_wait<true>(&sh.s_free[t], (v - 1) & 1, &sh.abort, &g_err_fwd);
            if (ok && !k_ready) {
              ok = wait_load(k_idx);
              k_ready = true;
            }
            if (!ok) break;
            tc_fence_after();
            issue_s(t, k_idx % C::kSlots);
          }
          // ... then PV_t(u) once the warpgroup wrote P_t(u) to its own columns.
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int u = j - j_lo[t];
            if (!ok || u < 0 || u >= len[t]) continue;
            if (!v_ready) {
              ok = wait_load(v_idx);
              v_ready = true;
            }
            if constexpr (C::kSplitP) {
              ok = ok && wait_p(&sh.p_half[t], u);
              if (!ok) break;
              tc_fence_after();
              issue_pv(t, v_idx % C::kSlots, u > 0, 0, C::kPVSteps / 2);
            }
            ok = ok && wait_p(&sh.p_full[t], u);
            if (!ok) break;
            tc_fence_after();
            issue_pv(t, v_idx % C::kSlots, u > 0, C::kSplitP ? C::kPVSteps / 2 : 0, C::kPVSteps);
            tc_commit(&sh.o_done[t]);
          }
        } else if constexpr (C::kSplitS) {
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (!ok) break;
            const int u = j - j_lo[t];
            const bool next = u + 1 >= 0 && u + 1 < len[t];
            // The first half of S_t(u+1) once the warpgroup has read S_t(u)'s first half ...
            if (next && u >= 0) {
              ok = mbar_wait<true>(&sh.s_free[t], u & 1, &sh.abort, &g_err_fwd);
              if (ok && !k_ready) {
                ok = wait_load(k_idx);
                k_ready = true;
              }
              if (!ok) break;
              tc_fence_after();
              issue_s_half(t, k_idx % C::kSlots, 0);
            }
            // ... PV_t(u) once it wrote P_t(u) over S_t(u)'s second half ...
            if (u >= 0 && u < len[t]) {
              if (!v_ready) {
                ok = wait_load(v_idx);
                v_ready = true;
              }
              if constexpr (C::kSplitP) {
                ok = ok && wait_p(&sh.p_half[t], u);
                if (!ok) break;
                tc_fence_after();
                issue_pv(t, v_idx % C::kSlots, u > 0, 0, C::kPVSteps / 2);
              }
              ok = ok && wait_p(&sh.p_full[t], u);
              if (!ok) break;
              tc_fence_after();
              issue_pv(t, v_idx % C::kSlots, u > 0, C::kSplitP ? C::kPVSteps / 2 : 0, C::kPVSteps);
              tc_commit(&sh.o_done[t]);
            }
            // ... and right behind it the second half of S_t(u+1) into P_t(u)'s
            // columns (both halves when the tile starts at block j + 1).
            if (next) {
              if (!k_ready) {
                ok = wait_load(k_idx);
                k_ready = true;
                if (!ok) break;
                tc_fence_after();
              }
              if (u + 1 == 0) issue_s_half(t, k_idx % C::kSlots, 0);
              issue_s_half(t, k_idx % C::kSlots, 1);
            }
          }
        } else {
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (!ok) break;
            const int u = j - j_lo[t];
            // PV_t(u) once the warpgroup wrote P_t(u) over S_t(u) ...
            if (u >= 0 && u < len[t]) {
              if (!v_ready) {
                ok = wait_load(v_idx);
                v_ready = true;
              }
              if constexpr (C::kSplitP) {  // keys 0-63 as soon as their P is there
                ok = ok && wait_p(&sh.p_half[t], u);
                if (!ok) break;
                tc_fence_after();
                issue_pv(t, v_idx % C::kSlots, u > 0, 0, C::kPVSteps / 2);
              }
              ok = ok && wait_p(&sh.p_full[t], u);
              if (!ok) break;
              tc_fence_after();
              issue_pv(t, v_idx % C::kSlots, u > 0, C::kSplitP ? C::kPVSteps / 2 : 0, C::kPVSteps);
              tc_commit(&sh.o_done[t]);
            }
            // ... and right behind it S_t(u+1) into the same columns.
            if (u + 1 >= 0 && u + 1 < len[t]) {
              if (!k_ready) {
                ok = wait_load(k_idx);
                k_ready = true;
                if (!ok) break;
                tc_fence_after();
              }
              issue_s(t, k_idx % C::kSlots);
            }
          }
        }
        if (!ok) break;
        if (k_ready) tc_commit(&sh.kv_empty[k_idx % C::kSlots]);
        if (v_ready) tc_commit(&sh.kv_empty[v_idx % C::kSlots]);
      }
      tc_commit(&sh.drain);
      mbar_wait_drain(&sh.drain, 0, &g_err_fwd);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;
    const int r = threadIdx.x & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t s_col = tmem + lane_base + C::kTmS + t * kBN;
    const uint32_t o_col = tmem + lane_base + C::kTmO + t * D;
    const uint32_t p_col = C::kEarlyS ? tmem + lane_base + C::kTmP + t * 64 : s_col + (C::kSplitS ? kBN / 2 : 0);
    const int row_g = q0 + t * kBM + r;
    const int jlo_t = t ? j_lo[1] : j_lo[0];
    const int nt = t ? len[1] : len[0];
    const int n64 = (N + 63) / 64;  // 64-key scale blocks (block-quantised K and V)
    float c = scale_log2;
    float o_mult = 1.0f;
    if constexpr (FP8 && !BS) {
      c = scale_log2 * __ldg(descale_q) * __ldg(descale_k);
      o_mult = __ldg(descale_v);
    }
    float cq = 0.f, inv_vmax = 1.f;
    const float* dk_row = nullptr;
    const float* dv_row = nullptr;
    if constexpr (BS) {
      dk_row = descale_k + static_cast<size_t>(bh_kv) * n64;
      dv_row = descale_v + static_cast<size_t>(bh_kv) * n64;
      if (nt > 0) {  // uniform over the warpgroup
        cq = scale_log2 * __ldg(descale_q + static_cast<size_t>(bh) * ((N + kBM - 1) / kBM) + q0 / kBM + t);
        float vm = 0.f;
        for (int jj = r; jj < n64; jj += kBM) vm = fmaxf(vm, __ldg(dv_row + jj));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) vm = fmaxf(vm, __shfl_xor_sync(0xffffffffu, vm, off));
        if ((r & 31) == 0) sh.vmax_part[t][warp & 3] = vm;
        named_bar_sync(1 + t, kBM);
        vm = fmaxf(fmaxf(sh.vmax_part[t][0], sh.vmax_part[t][1]), fmaxf(sh.vmax_part[t][2], sh.vmax_part[t][3]));
        o_mult = vm > 0.f ? vm : 1.0f;
        inv_vmax = 1.0f / o_mult;
      }
    }
    float m_used = -INFINITY;
    float l_sum = 0.0f;
    bool ok = true;
    for (int u = 0; u < nt; ++u) {
      const int j = jlo_t + u;
      // Scale factors of the two 64-key halves of this block (block-quantised
      // inputs: K's and V's scale blocks are 64 rows).
      float c0 = c, c1 = c, pm0 = 1.0f, pm1 = 1.0f;
      if constexpr (BS) {
        const int b0 = 2 * j, b1 = min(2 * j + 1, n64 - 1);
        c0 = cq * __ldg(dk_row + b0);
        c1 = cq * __ldg(dk_row + b1);
        pm0 = __ldg(dv_row + b0) * inv_vmax;
        pm1 = __ldg(dv_row + b1) * inv_vmax;
      }
      ok = mbar_wait<true>(&sh.s_full[t], u & 1, &sh.abort, &g_err_fwd);
      if (!ok) break;
      tc_fence_after();
      float s0[64], s1[64];
      const int key0 = j * kBN;
      const bool need_mask = (causal && key0 + kBN - 1 > q0 + t * kBM) || (key0 + kBN > N) ||
                             (WIN && key0 < q0 + t * kBM + kBM - window);
      const int lim = causal ? min(row_g, N - 1) : N - 1;  // last visible key
      const int lo = WIN ? row_g - window + 1 : 0;          // first visible key
      auto mask_half = [&](float (&sh_)[64], int k0) {
        if (need_mask) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (k0 + i > lim || (WIN && k0 + i < lo)) sh_[i] = -INFINITY;
        }
      };
      // Row maximum: independent chains of three-input maxima (measured against
      // two-input ones: +3 % at d = 128 without a mask, the same elsewhere),
      // then the block's candidate in log2 units (c0, c1 > 0 preserve the
      // order within each half).
      float mx[4];
      auto max_half = [&](const float (&sh_)[64], float& a, float& b) {
        a = sh_[0];
        b = sh_[1];
#pragma unroll
        for (int i = 2; i < 62; i += 4) {
          a = fmax3f(a, sh_[i], sh_[i + 2]);
          b = fmax3f(b, sh_[i + 1], sh_[i + 3]);
        }
        a = fmaxf(a, sh_[62]);
        b = fmaxf(b, sh_[63]);
      };
      if constexpr (C::kSplitS) {
        // First half: read, free its columns for S_t(u+1)'s first half, reduce;
        // then the second half, which follows PV_t(u-1) in issue order.
        {
          uint32_t ra[32], rb[32];
          tmem_ld32(s_col, ra);
          tmem_ld32(s_col + 32, rb);
          tmem_ld_wait(ra);
          tmem_ld_wait(rb);
          tc_fence_before();
          mbar_arrive(&sh.s_free[t]);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            s0[i] = __uint_as_float(ra[i]);
            s0[32 + i] = __uint_as_float(rb[i]);
          }
        }
        mask_half(s0, key0);
        max_half(s0, mx[0], mx[1]);
        ok = mbar_wait<true>(&sh.s_full_b[t], u & 1, &sh.abort, &g_err_fwd);
        if (!ok) break;
        tc_fence_after();
        {
          uint32_t rc[32], rd[32];
          tmem_ld32(s_col + 64, rc);
          tmem_ld32(s_col + 96, rd);
          tmem_ld_wait(rc);
          tmem_ld_wait(rd);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            s1[i] = __uint_as_float(rc[i]);
            s1[32 + i] = __uint_as_float(rd[i]);
          }
        }
        mask_half(s1, key0 + 64);
        max_half(s1, mx[2], mx[3]);
      } else {
        uint32_t ra[32], rb[32], rc[32], rd[32];
        tmem_ld32(s_col, ra);
        tmem_ld32(s_col + 32, rb);
        tmem_ld32(s_col + 64, rc);
        tmem_ld32(s_col + 96, rd);
        tmem_ld_wait(ra);
        tmem_ld_wait(rb);
        tmem_ld_wait(rc);
        tmem_ld_wait(rd);
        if constexpr (C::kEarlyS) {  // S_t's columns may take S_t(u+1) now
          tc_fence_before();
          mbar_arrive(&sh.s_free[t]);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          s0[i] = __uint_as_float(ra[i]);
          s0[32 + i] = __uint_as_float(rb[i]);
          s1[i] = __uint_as_float(rc[i]);
          s1[32 + i] = __uint_as_float(rd[i]);
        }
        mask_half(s0, key0);
        mask_half(s1, key0 + 64);
        mx[0] = s0[0];
        mx[1] = s0[1];
        mx[2] = s1[0];
        mx[3] = s1[1];
#pragma unroll
        for (int i = 2; i < 62; i += 4) {
          mx[0] = fmax3f(mx[0], s0[i], s0[i + 2]);
          mx[1] = fmax3f(mx[1], s0[i + 1], s0[i + 3]);
          mx[2] = fmax3f(mx[2], s1[i], s1[i + 2]);
          mx[3] = fmax3f(mx[3], s1[i + 1], s1[i + 3]);
        }
        mx[0] = fmaxf(mx[0], s0[62]);
        mx[1] = fmaxf(mx[1], s0[63]);
        mx[2] = fmaxf(mx[2], s1[62]);
        mx[3] = fmaxf(mx[3], s1[63]);
      }
      const float m_cand = fmaxf(fmaxf(mx[0], mx[1]) * c0, fmaxf(mx[2], mx[3]) * c1);
      float alpha = 1.0f;
      bool raise = false;
      if (u == 0) {
        m_used = m_cand;
      } else if (m_cand > m_used + C::kTauLog2) {
        raise = true;
        alpha = ex2_approx(m_used - m_cand);
        m_used = m_cand;
      }
      // A row with no visible key so far (only under a window) keeps m = -inf
      // and takes 0 as the exponent's reference: its p are all 0.
      const float m_ref = ((WIN && m_used == -INFINITY) ? 0.0f : m_used) + C::kPShiftLog2;
      // P over S_t: the first half's words go to the first columns (all of
      // S_t is in registers by now).
      // O_t may be rescaled once S_t(u) has completed (PV_t(u-1), issued before
      // it, is complete too), and must be before any PV_t(u): with P handed
      // over in halves, after the first half's P (when half of S is no longer
      // held in registers), else after both.
      auto rescale_o = [&]() {
        if (__any_sync(0xffffffffu, raise)) {
          // All 32-column loads in flight before one wait (FP8: S is no longer
          // held in registers here), two at a time when the second half of S is
          // (measured on inputs that raise often: +2.6 % FP8, +1 % bf16).
          constexpr int kG = C::kSplitP ? 2 : D / 32;
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32 * kG) {
            uint32_t rr[kG][32];
#pragma unroll
            for (int g = 0; g < kG; ++g) tmem_ld32(o_col + c0 + 32 * g, rr[g]);
#pragma unroll
            for (int g = 0; g < kG; ++g) tmem_ld_wait(rr[g]);
#pragma unroll
            for (int g = 0; g < kG; ++g) {
#pragma unroll
              for (int i = 0; i < 32; ++i) rr[g][i] = __float_as_uint(__uint_as_float(rr[g][i]) * alpha);
              tmem_st32(o_col + c0 + 32 * g, rr[g]);
            }
          }
        }
      };
      float row_sum;
      {
        uint32_t pw[C::kPWordsHalf];
        row_sum = exp2_pack_row<FP8, C::kEmuGroups, C::kPolyDeg, BS>(s0, c0, m_ref, pw, pm0);
        if constexpr (C::kEarlyS) {
          // P_t's columns and O_t are free once PV_t(u-1) has completed (with
          // P over S the completion of S_t(u) implied it).
          if (u > 0) {
            ok = mbar_wait<true>(&sh.o_done[t], (u - 1) & 1, &sh.abort, &g_err_fwd);
            if (!ok) break;
            tc_fence_after();
          }
        }
        if constexpr (FP8) tmem_st16(p_col, pw);
        else tmem_st32(p_col, pw);
      }
      if constexpr (C::kSplitP) {  // keys 0-63 handed over
        rescale_o();
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sh.p_half[t]);
      }
      {
        uint32_t pw[C::kPWordsHalf];
        row_sum += exp2_pack_row<FP8, C::kEmuGroups, C::kPolyDeg, BS>(s1, c1, m_ref, pw, pm1);
        if constexpr (FP8) tmem_st16(p_col + 16, pw);
        else tmem_st32(p_col + 32, pw);
      }
      if constexpr (!C::kSplitP) rescale_o();  // (after both halves: no S left in registers)
      l_sum = l_sum * alpha + row_sum;
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sh.p_full[t]);
    }
    // Epilogue: O = O~ / l in bf16, staged with the 128-byte swizzle in this
    // tile's own Q space and written by TMA stores, which drop box rows past N.
    // The Q tile is dead here: the MMA thread issued the tile's last S product
    // before its last PV, so the o_done completion covers it.  Every thread of
    // the warpgroup takes every barrier below, so a failed wait in one of them
    // cannot leave the others waiting; a store is issued only if all were fine.
    if (nt > 0) {
      if (ok) {
        ok = mbar_wait<true>(&sh.o_done[t], (nt - 1) & 1, &sh.abort, &g_err_fwd);
        tc_fence_after();
      }
      const float inv = o_mult / l_sum;
      uint8_t* stage = s_q + t * C::kTileBytes;
      const int ro = r % C::kORows;  // row within a staged group
      const uint32_t sw = static_cast<uint32_t>(ro & 7);
      const bool leader = r == 0;
      constexpr int kStage = C::kOStageBlocks < C::kOColBlocks ? C::kOStageBlocks : C::kOColBlocks;
      int round = 0;
#pragma unroll 1
      for (int rg = 0; rg < kBM / C::kORows; ++rg) {
#pragma unroll 1
        for (int ob = 0; ob < C::kOColBlocks; ob += kStage, ++round) {
          if (round > 0) {  // the staging space is reused: earlier stores must have read it
            if (leader) bulk_wait_read_all();
            named_bar_sync(1 + t, kBM);
          }
          if (ok && r / C::kORows == rg) {
#pragma unroll
            for (int b = 0; b < kStage; ++b) {
              uint8_t* row_base = stage + b * C::kOStageBytes + ro * 128;
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                uint32_t rr[32];
                tmem_ld32(o_col + (ob + b) * 64 + h * 32, rr);
                tmem_ld_wait(rr);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                  pk[i] = pack_bf16x2(__uint_as_float(rr[2 * i]) * inv, __uint_as_float(rr[2 * i + 1]) * inv);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  *reinterpret_cast<uint4*>(row_base + (((h * 4 + i) ^ sw) << 4)) =
                      make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
              }
            }
            fence_proxy_async_smem();
          }
          ok = named_bar_and(1 + t, kBM, ok);
          if (ok && leader) {
#pragma unroll
            for (int b = 0; b < kStage; ++b)
              tma_store_3d(&map_o, (ob + b) * 64, q0 + t * kBM + rg * C::kORows, bh, stage + b * C::kOStageBytes);
            bulk_commit_group();
          }
        }
      }
      if (leader) bulk_wait_read_all();
      if (ok && row_g < N)
        out_lse[static_cast<size_t>(bh) * N + row_g] = (m_used + C::kPShiftLog2) * 0.69314718055994531f + logf(l_sum);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool FP8, bool BS, bool WIN>
fa_status launch_fwd_impl(const FwdArgs& a, cudaStream_t stream) {
  using C = FwdCfg<D, FP8>;
  const int BH = a.B * a.H;
  const int BHkv = a.B * a.Hkv;
  CUtensorMap mq, mk, mv, mo;
  if (!encode_rows_map(&mq, a.q, C::kElemBytes, D, a.N, BH, C::kBoxCols, kBM, C::kSwz) ||
      !encode_rows_map(&mo, a.o, 2, D, a.N, BH, 64, C::kORows) ||
      !encode_rows_map(&mk, a.k, C::kElemBytes, D, a.N, BHkv, C::kBoxCols, kBN, C::kSwz) ||
      !encode_rows_map(&mv, a.v, C::kElemBytes, D, a.N, BHkv, C::kBoxCols, kBN, C::kSwz))
    return FA_ERR_LAUNCH;
  auto kern = fa_fwd_kernel<D, FP8, BS, WIN>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
    return FA_ERR_LAUNCH;
  dim3 grid(static_cast<unsigned>(((a.N + 2 * kBM - 1) / (2 * kBM)) * BH));
  const float scale_log2 = a.scale * 1.4426950408889634f;
  const int qgroup = a.H / a.Hkv;
  const long long kv_bytes_per_qhead = 2ll * a.N * D * C::kElemBytes / qgroup;
  int group = static_cast<int>(std::max<long long>(1, (32ll << 20) / std::max<long long>(1, kv_bytes_per_qhead)));
  group = std::min(group, BH);
  const cudaError_t e = launch_pdl(kern, grid, dim3(kThreads), C::kSmemBytes, stream, mq, mk, mv, mo, a.lse,
                                   a.descale_q, a.descale_k, a.descale_v, BH, a.N, a.causal, scale_log2, a.H, qgroup,
                                   a.window, group);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

fa_status launch_fwd_bf16(const FwdArgs& a, cudaStream_t stream) {
  if (a.window > 0)
    return a.d == 64 ? launch_fwd_impl<64, false, false, true>(a, stream)
                     : launch_fwd_impl<128, false, false, true>(a, stream);
  return a.d == 64 ? launch_fwd_impl<64, false, false, false>(a, stream)
                   : launch_fwd_impl<128, false, false, false>(a, stream);
}

fa_status launch_fwd_fp8(const FwdArgs& a, cudaStream_t stream) {
  return a.d == 64 ? launch_fwd_impl<64, true, false, false>(a, stream)
                   : launch_fwd_impl<128, true, false, false>(a, stream);
}

fa_status launch_fwd_fp8_blocks(const FwdArgs& a, cudaStream_t stream) {
  return a.d == 64 ? launch_fwd_impl<64, true, true, false>(a, stream)
                   : launch_fwd_impl<128, true, true, false>(a, stream);
}

uint32_t fwd_bf16_take_error(cudaStream_t s) {
  uint32_t v = 0, zero = 0;
  cudaMemcpyFromSymbolAsync(&v, g_err_fwd, sizeof(v), 0, cudaMemcpyDeviceToHost, s);
  cudaStreamSynchronize(s);
  cudaMemcpyToSymbolAsync(g_err_fwd, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
  cudaStreamSynchronize(s);
  return v;
}

uint32_t fwd_fp8_take_error(cudaStream_t) { return 0; }  // shares the word above

}  // namespace fa
