// Backward attention kernels for sm_103a.
//
// The chain rule for O = softmax(S) V, S = scale * Q K^T ("FLASH-ATTN",
// FlashAttention-2 > Background): dV = P^T dO, dP = dO V^T, dS = P o (dP - D)
// with D_i = sum_j P_ij dP_ij (the row-softmax Jacobian), dQ = scale dS K,
// dK = scale dS^T Q.  P is rebuilt block by block from the saved L
// (P_ij = exp(S_ij - L_i)) instead of being stored ("FLASH-ATTN",
// FlashAttention > Tiling and Recomputation: selective recomputation).
//
// Three kernels:
//  1. fa_bwd_preprocess: D_i = sum_k dO_ik O_ik (equal to sum_j P_ij dP_ij
//     because O = P V) and zeros for the fp32 dQ accumulator.  HBM bound.
//  2. fa_bwd_main_kernel: one CTA per 128-key block of a head, query blocks
//     inner ("FLASH-ATTN", FlashAttention-2 > Parallelism: column blocks get
//     their own thread blocks and meet only through atomic adds to dQ).  The
//     five products run on tcgen05 with accumulators in TMEM:
//       S^T  = K Q_i^T        (smem x smem)        -> TMEM
//       dP^T = V dO_i^T       (smem x smem)        -> TMEM
//       dV  += P^T dO_i       (P^T from TMEM)      -> TMEM, whole loop
//       dK  += dS^T Q_i       (dS^T from smem)     -> TMEM, whole loop
//       dQ_i = dS K           (dS^T read MN-major) -> TMEM, then TMA reduce-adds
//                                                     into an fp32 accumulator
//     Causal: query blocks below the key block are skipped; only the
//     diagonal block applies the element mask.
//  3. fa_bwd_dq_convert: dQ = bf16(scale * dQ_acc).  HBM bound.
//
// Roles of fa_bwd_main_kernel (512 threads, four warpgroups):
//  warps 0-3  thread r owns key row r for queries 0-63 of the block:
//             P^T = exp2(S^T c - L_i log2 e) into TMEM (bf16; over S^T at d = 128), then
//             dS^T = P^T o (dP^T - D_i) into smem; finally half of dV (TMA store).
//  warps 12-15 the same for queries 64-127 and the other half of dV.
//  warps 4-7  thread r owns query row r of the current block: reads dQ_i
//             from TMEM and adds it into the fp32 accumulator; finally
//             writes dK = scale * acc (TMA store).
//  warp 8     TMA producer: K and V once, Q_i into two stages, dO_i into one
//             (d = 64: three and two).
//  warp 9     TMEM allocation and the single MMA-issuing thread.
//  warp 10    L_i and D_i of each query block into shared memory (two stages).
//  warp 11    no role (it completes the TMA/MMA warpgroup).
//
// Per query block the MMA thread issues, at d = 128, dV_i, S_(i+1), dK_i,
// dQ_i, dP_(i+1) (dQ_i shares dP^T's TMEM columns); at d = 64, where S^T, P^T,
// dP^T and dQ each have columns of their own, dV_i and S_(i+1), then
// dP_(i+1) as soon as the key rows have read dP_i, then dK_i and dQ_i, so that
// the next S and dP are ready before the key rows need them.
#include <cuda_bf16.h>

#include <algorithm>

#include "fa_common.cuh"
#include "fa_host.h"

namespace fa {

namespace {

__device__ uint32_t g_err_bwd;

constexpr int kThreads = 512;
// Registers per thread at launch: 512 threads leave 128 each.  The build
// checks that the compiled d = 128 kernels use exactly this many, and the
// launcher checks it again (FA_ERR_KERNEL_CONFIG otherwise), because the
// setmaxnreg split below must add up to the launch allocation.
constexpr int kRegLaunch = 128;
constexpr float kLog2e = 1.4426950408889634f;
// Rows (B * H * N) up to which the preprocess and convert kernels are launched
// with programmatic stream serialization (see launch_bwd_preprocess).
constexpr long long kSmallRows = 65536;

// ---------------------------------------------------------------- preprocess

template <int D>
__global__ void __launch_bounds__(256) fa_bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ o,
                                                                const __nv_bfloat16* __restrict__ dout,
                                                                float* __restrict__ dvec,
                                                                float* __restrict__ dq_acc, long long rows) {
  pdl_launch_dependents();
  pdl_wait_prior();
  constexpr int kLanesPerRow = D / 8;  // each lane: 8 bf16 = 16 bytes of O and of dO
  constexpr int kRowsPerBlock = 256 / kLanesPerRow;
  const int sub = threadIdx.x % kLanesPerRow;
  const long long row = static_cast<long long>(blockIdx.x) * kRowsPerBlock + threadIdx.x / kLanesPerRow;
  float acc = 0.f;
  if (row < rows) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(o + row * D) + sub);
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(dout + row * D) + sub);
    const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 fa_ = __bfloat1622float2(pa[i]);
      const float2 fb_ = __bfloat1622float2(pb[i]);
      acc = fmaf(fa_.x, fb_.x, acc);
      acc = fmaf(fa_.y, fb_.y, acc);
    }
    float4* z = reinterpret_cast<float4*>(dq_acc + row * D) + 2 * sub;
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int off = kLanesPerRow / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (row < rows && sub == 0) dvec[row] = acc;
}

// ---------------------------------------------------------------- convert

__global__ void __launch_bounds__(256) fa_bwd_dq_convert_kernel(const float* __restrict__ acc,
                                                                __nv_bfloat16* __restrict__ dq, long long n8,
                                                                float scale) {
  pdl_launch_dependents();
  pdl_wait_prior();
  // Groups of 8 values; each thread keeps four groups' loads in flight before
  // converting and storing them.  Both streams are touched once: loads and
  // stores marked evict-first (measured: 35.3 -> 32.8 us on the long causal
  // workload's 134 MB accumulator).
  constexpr int kU = 4;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + (kU - 1) * stride < n8; i += kU * stride) {
    float4 a[kU], b[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      a[u] = __ldcs(reinterpret_cast<const float4*>(acc) + 2 * (i + u * stride));
      b[u] = __ldcs(reinterpret_cast<const float4*>(acc) + 2 * (i + u * stride) + 1);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      uint4 r;
      r.x = pack_bf16x2(a[u].x * scale, a[u].y * scale);
      r.y = pack_bf16x2(a[u].z * scale, a[u].w * scale);
      r.z = pack_bf16x2(b[u].x * scale, b[u].y * scale);
      r.w = pack_bf16x2(b[u].z * scale, b[u].w * scale);
      __stcs(reinterpret_cast<uint4*>(dq) + i + u * stride, r);
    }
  }
  for (; i < n8; i += stride) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(acc) + 2 * i);
    const float4 b = __ldg(reinterpret_cast<const float4*>(acc) + 2 * i + 1);
    uint4 r;
    r.x = pack_bf16x2(a.x * scale, a.y * scale);
    r.y = pack_bf16x2(a.z * scale, a.w * scale);
    r.z = pack_bf16x2(b.x * scale, b.y * scale);
    r.w = pack_bf16x2(b.z * scale, b.w * scale);
    reinterpret_cast<uint4*>(dq)[i] = r;
  }
}

// ---------------------------------------------------------------- main

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = 128 * D * 2;   // one 128-row bf16 tile
  static constexpr int kColBlocks = D / 64;        // 128-byte column blocks per bf16 row
  static constexpr int kBlockBytes = 128 * 128;    // one 128-row x 128-byte block
  static constexpr int kDsBytes = 128 * 128 * 2;   // dS^T, 128 keys x 128 queries, bf16
  static constexpr int kStageBytes = 32768;        // dQ staging: 2 blocks of 128 rows x 32 fp32, used in turn
  // shared memory layout (offsets from a 1024-aligned base)
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kTileBytes;
  // At d = 64 the next block's dP^T is issued as soon as the key rows have read
  // this block's, and the next S^T right behind dV (their TMEM columns are not
  // shared with P or dQ there); shared memory has room for the copies that
  // feeds: three Q and two dO stages (measured: +6-7 % on the d = 64 backward
  // at N = 8192 and 16384, +1-4 % at N = 512 and 1024).  A second dS^T buffer
  // measured the same or slower.
  static constexpr bool kEarly = (D == 64);
  static constexpr int kQStages = kEarly ? 3 : 2;
  static constexpr int kDoStages = kEarly ? 2 : 1;
  static constexpr int kOffQ = kOffV + kTileBytes;                  // kQStages stages
  static constexpr int kOffDO = kOffQ + kQStages * kTileBytes;      // kDoStages stages
  static constexpr int kOffDS = kOffDO + kDoStages * kTileBytes;
  static constexpr int kOffStage = kOffDS + kDsBytes;
  static constexpr int kOffL = kOffStage + kStageBytes;      // float [2][128]
  static constexpr int kOffDv = kOffL + 2 * 128 * 4;         // float [2][128]
  static constexpr int kOffBar = kOffDv + 2 * 128 * 4;
  static constexpr int kSmemBytes = kOffBar + 256;
  // TMEM columns
  static constexpr uint32_t kTmDV = 0;
  static constexpr uint32_t kTmDK = D;
  static constexpr uint32_t kTmS = 2 * D;
  static constexpr uint32_t kTmDP = 2 * D + 128;
  static constexpr uint32_t kTmDQ = (D == 128) ? kTmDP : 2 * D + 256;  // aliases dP^T when D = 128
  // P^T (bf16 pairs, 64 columns): at d = 64 in the spare columns 448-511, so
  // that S^T of the next block need not wait for dV to have read P; at d = 128
  // over S^T (queries 0-63 in columns 0-31, 64-127 in 96-127).
  static constexpr bool kOwnP = (D == 64);
  static constexpr uint32_t kTmP = kOwnP ? 2 * D + 256 + 64 : kTmS;
  static_assert(!kOwnP || kTmP + 64 <= 512, "TMEM columns");
  static constexpr uint32_t kIdescKK = idesc_bf16(128, 128, false, false);
  static constexpr uint32_t kIdescKM = idesc_bf16(128, D, false, true);
  static constexpr uint32_t kIdescMM = idesc_bf16(128, D, true, true);
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // Registers per thread after the warpgroups' setmaxnreg: at d = 128 the dQ
  // warpgroup holds a whole 128-column fp32 dQ row, so it takes registers from
  // the key-row and TMA/MMA warpgroups; the four shares add up to the launch
  // allocation (a larger sum would leave the increase waiting forever).
  static constexpr bool kRegSplit = (D == 128);
  static constexpr int kRegKeyRow = kRegSplit ? 120 : kRegLaunch;
  static constexpr int kRegCtl = kRegSplit ? 96 : kRegLaunch;
  static constexpr int kRegDq = kRegSplit ? 176 : kRegLaunch;
  static_assert(2 * kRegKeyRow + kRegCtl + kRegDq == 4 * kRegLaunch, "register split");
};

template <int D>
struct BwdBars {
  uint64_t kv_full;
  uint64_t q_full[BwdCfg<D>::kQStages];
  uint64_t q_empty[BwdCfg<D>::kQStages];
  uint64_t do_full[BwdCfg<D>::kDoStages], do_empty[BwdCfg<D>::kDoStages];
  uint64_t ld_full[2];
  uint64_t ld_empty[2];
  uint64_t s_full, p_ready, dp_full, ds_ready, dq_full, dq_free, acc_done, drain;
  uint32_t tmem_base;
  CtaAbort abort;
  uint64_t dp_free;  // d = 64 only
};

// Block index -> (head, key block).  Heads are taken in groups whose Q, dO
// and dQ accumulator fit in L2 together; within a group the key blocks with
// the most query blocks (causal: the lowest) come first.  A partial group (the
// remainder of BH / group) goes first, so that every later group runs long
// enough to absorb its own heaviest blocks and the launch ends on light ones.
__device__ __forceinline__ void bwd_item(int item, int BH, int n_blk, int group, int& bh, int& kb) {
  const int rem = BH % group;
  int g_heads, base_item, base_head;
  if (item < rem * n_blk) {
    g_heads = rem;
    base_item = 0;
    base_head = 0;
  } else {
    const int g = (item - rem * n_blk) / (group * n_blk);
    g_heads = group;
    base_item = rem * n_blk + g * group * n_blk;
    base_head = rem + g * group;
  }
  const int r = item - base_item;
  kb = r / g_heads;
  bh = base_head + (r - kb * g_heads);
}

// WIN: causal sliding window of `window` keys.  SPLIT (grouped-query heads):
// one CTA per (query head, key block) instead of per (key/value head, key
// block); each CTA adds its partial dK and dV (fp32) into accumulators of the
// key/value head by TMA reduce-adds, so a group's query heads run in parallel.
template <int D, bool WIN, bool SPLIT = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_bwd_main_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                       const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
                       const __grid_constant__ CUtensorMap map_dq, const __grid_constant__ CUtensorMap map_dk,
                       const __grid_constant__ CUtensorMap map_dv, const float* __restrict__ lse,
                       const float* __restrict__ dvec, int BH, int N, int causal, float scale,
                       float scale_log2, int head_group, int H, int qgroup, int window) {
  using C = BwdCfg<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  static_assert(sizeof(BwdBars<D>) <= 256, "barrier block");
  BwdBars<D>& sh = *reinterpret_cast<BwdBars<D>*>(smem + C::kOffBar);
  // The tile offsets assume a 1024-byte aligned base (the swizzle atoms).
  if ((smem_u32(smem) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(&g_err_bwd, 2u);
    return;
  }

  float* s_lse2 = reinterpret_cast<float*>(smem + C::kOffL);
  float* s_dvec = reinterpret_cast<float*>(smem + C::kOffDv);

  const int warp = warp_id();
  const int n_blk = (N + 127) / 128;
  // bh: the K/V head of this CTA (BH of them); its query heads are the
  // `qgroup` consecutive heads qh0 .. qh0 + qgroup - 1 (grouped-query
  // attention; qgroup = 1 when every query head has its own K/V head).  With
  // SPLIT the items are query heads (BH of them) and bh is derived: the CTA
  // takes one query head, qh0, of the K/V head bh.
  int item_h, kb;
  bwd_item(static_cast<int>(blockIdx.x), BH, n_blk, head_group, item_h, kb);
  const int hkv = H / qgroup;
  const int bh = SPLIT ? (item_h / H) * hkv + (item_h % H) / qgroup : item_h;
  const int qh0 = SPLIT ? item_h : (bh / hkv) * H + (bh % hkv) * qgroup;
  const int heads = SPLIT ? 1 : qgroup;  // query heads this CTA walks
  const int i_begin = causal ? kb : 0;
  // With a sliding window of `window` keys (causal), the last query that sees
  // key kb*128 + 127 is kb*128 + 126 + window.
  const int i_end = WIN ? min(n_blk, (kb * 128 + 126 + window) / 128 + 1) : n_blk;
  const int n_per = i_end - i_begin;  // query blocks per query head
  const int n_it = heads * n_per;
  // Every role walks the same (query head, query block) sequence: query
  // blocks i_begin .. i_end-1 of head qh0, then of qh0 + 1, and so on.
  struct QCursor {
    int i, h;
  };
  auto q_advance = [&](QCursor& c, int it) {
    if (it > 0 && ++c.i == i_end) {
      c.i = i_begin;
      ++c.h;
    }
  };

  if (threadIdx.x == 0) {
    // A wait of an earlier CTA ran out: the launch is already failed, and this
    // CTA stops after its set-up (the word stays set until fa_device_error
    // reads and clears it).  The load's latency overlaps the set-up.
    const uint32_t err0 = *reinterpret_cast<volatile uint32_t*>(&g_err_bwd);
    mbar_init(&sh.kv_full, 1);
    for (int s = 0; s < C::kQStages; ++s) {
      mbar_init(&sh.q_full[s], 1);
      mbar_init(&sh.q_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sh.ld_full[s], 32);
      mbar_init(&sh.ld_empty[s], 256);
    }
    for (int s = 0; s < C::kDoStages; ++s) {
      mbar_init(&sh.do_full[s], 1);
      mbar_init(&sh.do_empty[s], 1);
    }
    mbar_init(&sh.dp_free, 256);
    mbar_init(&sh.s_full, 1);
    mbar_init(&sh.p_ready, 256);
    mbar_init(&sh.dp_full, 1);
    mbar_init(&sh.ds_ready, 256);
    mbar_init(&sh.dq_full, 1);
    mbar_init(&sh.dq_free, 128);
    mbar_init(&sh.acc_done, 1);
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

  if (warp >= 8 && warp < 12) {
    // TMA/MMA warpgroup: warp 8 issues the tile copies, warp 9 the products,
    // warp 10 loads L and D; warp 11 has no role.
    if constexpr (C::kRegSplit) setmaxnreg_dec<C::kRegCtl>();
    if (warp == 8) {
      // ------------------------------------------------------------ producer
      const int lane = lane_id();
      if (lane == 0) {
        tma_prefetch_desc(&map_q);
        tma_prefetch_desc(&map_do);
        mbar_arrive_expect_tx(&sh.kv_full, 2 * C::kTileBytes);
        for (int cb = 0; cb < C::kColBlocks; ++cb) {
          tma_load_3d(smem + C::kOffK + cb * C::kBlockBytes, &map_k, cb * 64, kb * 128, bh, &sh.kv_full);
          tma_load_3d(smem + C::kOffV + cb * C::kBlockBytes, &map_v, cb * 64, kb * 128, bh, &sh.kv_full);
        }
      }
      int q_issued[C::kQStages] = {};
      int do_issued[C::kDoStages] = {};
      QCursor cur{i_begin, qh0};
      for (int it = 0; it < n_it; ++it) {
        q_advance(cur, it);
        if (__shfl_sync(0xffffffffu, sh.abort.flag, 0)) break;  // one decision for the whole warp
        const int st = it % C::kQStages;
        const int use = it / C::kQStages;
        const int sd = it % C::kDoStages;
        const int used = it / C::kDoStages;
        const int qrow0 = cur.i * 128;
        const int qh = cur.h;
        bool ok = true;
        if (lane == 0) {
          // Q_i: kQStages stages, each freed when the dK that read it is done.
          if (use > 0) ok = mbar_wait(&sh.q_empty[st], (use - 1) & 1, &sh.abort, &g_err_bwd);
          if (ok) {
            mbar_arrive_expect_tx(&sh.q_full[st], C::kTileBytes);
            for (int cb = 0; cb < C::kColBlocks; ++cb)
              tma_load_3d(smem + C::kOffQ + st * C::kTileBytes + cb * C::kBlockBytes, &map_q, cb * 64, qrow0, qh,
                          &sh.q_full[st]);
            ++q_issued[st];
          }
          // dO_i: kDoStages stages, each freed when the dV that read it is done.
          if (ok && used > 0) ok = mbar_wait(&sh.do_empty[sd], (used - 1) & 1, &sh.abort, &g_err_bwd);
          if (ok) {
            mbar_arrive_expect_tx(&sh.do_full[sd], C::kTileBytes);
            for (int cb = 0; cb < C::kColBlocks; ++cb)
              tma_load_3d(smem + C::kOffDO + sd * C::kTileBytes + cb * C::kBlockBytes, &map_do, cb * 64, qrow0, qh,
                          &sh.do_full[sd]);
            ++do_issued[sd];
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
      if (lane == 0 && sh.abort.flag) {
        // Let every copy still in flight land before the CTA's memory goes away.
        mbar_wait_drain(&sh.kv_full, 0, &g_err_bwd);
        for (int s2 = 0; s2 < C::kQStages; ++s2)
          if (q_issued[s2] > 0) mbar_wait_drain(&sh.q_full[s2], (q_issued[s2] - 1) & 1, &g_err_bwd);
        for (int s2 = 0; s2 < C::kDoStages; ++s2)
          if (do_issued[s2] > 0) mbar_wait_drain(&sh.do_full[s2], (do_issued[s2] - 1) & 1, &g_err_bwd);
      }
      __syncwarp();
    } else if (warp == 9) {
      // ------------------------------------------------------------ MMA issuer
      // Per query block i the five products are issued as
      //   dV_i, S_(i+1), dK_i, dQ_i, dP_(i+1)
      // so the key-row warpgroup computes P_(i+1) while dK_i and dQ_i run.
      if (elect_one()) {
        const uint32_t sm = smem_u32(smem);
        // Base descriptors (K-major "_k", MN-major "_mn"); operands below advance
        // them by byte offsets that are compile-time constants after unrolling.
        const uint64_t k_k = sdesc_sw128(sm + C::kOffK, 16, 1024), k_mn = sdesc_sw128(sm + C::kOffK, C::kBlockBytes, 1024);
        const uint64_t v_k = sdesc_sw128(sm + C::kOffV, 16, 1024);
        const uint64_t ds_k = sdesc_sw128(sm + C::kOffDS, 16, 1024), ds_mn = sdesc_sw128(sm + C::kOffDS, C::kBlockBytes, 1024);
        const uint64_t do_k = sdesc_sw128(sm + C::kOffDO, 16, 1024), do_mn = sdesc_sw128(sm + C::kOffDO, C::kBlockBytes, 1024);
        const uint64_t q_k = sdesc_sw128(sm + C::kOffQ, 16, 1024), q_mn = sdesc_sw128(sm + C::kOffQ, C::kBlockBytes, 1024);
        auto issue_s = [&](int i) {  // S^T = K Q_i^T
          const uint64_t qb = sdesc_advance(q_k, (i % C::kQStages) * C::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kBlockBytes + (kk & 3) * 32;
            mma_bf16_ss(tmem + C::kTmS, sdesc_advance(k_k, off), sdesc_advance(qb, off), C::kIdescKK, kk > 0);
          }
          tc_commit(&sh.s_full);
        };
        auto issue_dp = [&](int i) {  // dP^T = V dO_i^T
          const uint64_t db = sdesc_advance(do_k, (i % C::kDoStages) * C::kTileBytes);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * C::kBlockBytes + (kk & 3) * 32;
            mma_bf16_ss(tmem + C::kTmDP, sdesc_advance(v_k, off), sdesc_advance(db, off), C::kIdescKK, kk > 0);
          }
          tc_commit(&sh.dp_full);
        };
        bool ok = mbar_wait(&sh.kv_full, 0, &sh.abort, &g_err_bwd) &&
                  mbar_wait(&sh.q_full[0], 0, &sh.abort, &g_err_bwd);
        if (ok) {
          tc_fence_after();
          issue_s(0);
          ok = mbar_wait(&sh.do_full[0], 0, &sh.abort, &g_err_bwd);
          if (ok) {
            tc_fence_after();
            issue_dp(0);
          }
        }
        for (int it = 0; ok && it < n_it; ++it) {
          const int st = it % C::kQStages;
          const uint64_t qm = sdesc_advance(q_mn, st * C::kTileBytes);
          const uint64_t dom = sdesc_advance(do_mn, (it % C::kDoStages) * C::kTileBytes);
          const bool has_next = it + 1 < n_it;
          if constexpr (C::kEarly) {
            // dV_i once the key rows wrote P_i ...
            ok = mbar_wait(&sh.p_ready, it & 1, &sh.abort, &g_err_bwd);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_bf16_ts(tmem + C::kTmDV, tmem + C::kTmP + kk * 8, sdesc_advance(dom, kk * 2048), C::kIdescKM,
                          (it > 0 || kk > 0) ? 1u : 0u);
            tc_commit(&sh.do_empty[it % C::kDoStages]);
            // ... S_(i+1) right behind it (the key rows read S_i before writing
            // P_i; issued after dV_i, its completion, which they await before
            // writing P_(i+1), covers dV_i's reads of P_i) ...
            if (has_next) {
              ok = mbar_wait(&sh.q_full[(it + 1) % C::kQStages], ((it + 1) / C::kQStages) & 1, &sh.abort, &g_err_bwd);
              if (!ok) break;
              tc_fence_after();
              issue_s(it + 1);
            }
            // ... dP_(i+1) once they have read dP_i ...
            if (has_next) {
              ok = mbar_wait(&sh.dp_free, it & 1, &sh.abort, &g_err_bwd) &&
                   mbar_wait(&sh.do_full[(it + 1) % C::kDoStages], ((it + 1) / C::kDoStages) & 1, &sh.abort,
                             &g_err_bwd);
              if (!ok) break;
              tc_fence_after();
              issue_dp(it + 1);
            }
            // ... and dK_i, dQ_i once they wrote dS_i (dQ_i after the read-out of dQ_(i-1)).
            ok = mbar_wait(&sh.ds_ready, it & 1, &sh.abort, &g_err_bwd);
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t off = (kk >> 2) * C::kBlockBytes + (kk & 3) * 32;
              mma_bf16_ss(tmem + C::kTmDK, sdesc_advance(ds_k, off), sdesc_advance(qm, kk * 2048), C::kIdescKM,
                          (it > 0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(&sh.q_empty[st]);
            if (it > 0) {
              ok = mbar_wait(&sh.dq_free, (it - 1) & 1, &sh.abort, &g_err_bwd);
              if (!ok) break;
              tc_fence_after();
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_bf16_ss(tmem + C::kTmDQ, sdesc_advance(ds_mn, kk * 2048), sdesc_advance(k_mn, kk * 2048), C::kIdescMM,
                          kk > 0);
            tc_commit(&sh.dq_full);
            continue;
          }
          // dV += P_i^T dO_i
          ok = mbar_wait(&sh.p_ready, it & 1, &sh.abort, &g_err_bwd);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ts(tmem + C::kTmDV, tmem + C::kTmP + kk * 8 + ((C::kOwnP || kk < 4) ? 0 : 64),
                        sdesc_advance(dom, kk * 2048), C::kIdescKM, (it > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&sh.do_empty[it % C::kDoStages]);
          // S_(i+1): at d = 128 its columns hold P_i^T, which dV_i reads.  The
          // tcgen05.mma operations of one thread execute in issue order, so
          // S_(i+1) issued right behind dV_i overwrites P_i^T only after dV_i
          // has read it (measured: +0.5 % over waiting for dV_i to complete).
          if (has_next) {
            ok = mbar_wait(&sh.q_full[(it + 1) % C::kQStages], ((it + 1) / C::kQStages) & 1, &sh.abort, &g_err_bwd);
            if (!ok) break;
            tc_fence_after();
            issue_s(it + 1);
          }
          // dK += dS_i^T Q_i ; dQ_i = dS_i K
          ok = mbar_wait(&sh.ds_ready, it & 1, &sh.abort, &g_err_bwd);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * C::kBlockBytes + (kk & 3) * 32;
            mma_bf16_ss(tmem + C::kTmDK, sdesc_advance(ds_k, off), sdesc_advance(qm, kk * 2048), C::kIdescKM,
                        (it > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&sh.q_empty[st]);
          if (D == 64 && it > 0) {  // separate dQ columns: only the previous read-out must be done
            ok = mbar_wait(&sh.dq_free, (it - 1) & 1, &sh.abort, &g_err_bwd);
            if (!ok) break;
            tc_fence_after();
          }
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_bf16_ss(tmem + C::kTmDQ, sdesc_advance(ds_mn, kk * 2048), sdesc_advance(k_mn, kk * 2048), C::kIdescMM,
                        kk > 0);
          tc_commit(&sh.dq_full);
          // dP_(i+1)
          if (has_next) {
            ok = mbar_wait(&sh.do_full[(it + 1) % C::kDoStages], ((it + 1) / C::kDoStages) & 1, &sh.abort, &g_err_bwd);
            if (ok && D == 128)  // dP^T shares columns with dQ_i
              ok = mbar_wait(&sh.dq_free, it & 1, &sh.abort, &g_err_bwd);
            if (!ok) break;
            tc_fence_after();
            issue_dp(it + 1);
          }
        }
        if (ok) tc_commit(&sh.acc_done);
        tc_commit(&sh.drain);
        mbar_wait_drain(&sh.drain, 0, &g_err_bwd);
      }
      __syncwarp();
    } else if (warp == 10) {
      // ------------------------------------------------------------ L and D rows
      // L in log2 units (+inf past the end: P = 0 there) and D of each query
      // block, two stages ahead of the key-row warpgroups, 4 rows per lane.
      const int lane = lane_id();
      QCursor cur{i_begin, qh0};
      for (int it = 0; it < n_it; ++it) {
        q_advance(cur, it);
        const int st = it & 1;
        const int use = it >> 1;
        if (use > 0 && !mbar_wait(&sh.ld_empty[st], (use - 1) & 1, &sh.abort, &g_err_bwd)) break;
        const int qrow0 = cur.i * 128;
        const int qh = cur.h;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int r = lane * 4 + u;
          const int qg = qrow0 + r;
          float l2 = -INFINITY, dd = -0.f;  // stored negated: -L log2 e and -D
          if (qg < N) {
            l2 = __ldg(lse + static_cast<size_t>(qh) * N + qg) * -kLog2e;
            dd = -__ldg(dvec + static_cast<size_t>(qh) * N + qg);
          }
          s_lse2[st * 128 + r] = l2;
          s_dvec[st * 128 + r] = dd;
        }
        mbar_arrive(&sh.ld_full[st]);
      }
    }
  } else if (warp < 4 || warp >= 12) {
    // ------------------------------------------------------------ P and dS (key rows)
    // Two warpgroups share the key rows: warps 0-3 take queries 0-63 of the
    // block, warps 12-15 queries 64-127 (a warp reaches the TMEM lanes of its
    // own quarter, warp % 4).  At d = 128, P^T of the first half goes to
    // S^T's columns 0-31 and of the second to columns 96-127, columns that
    // each warpgroup has already read itself; at d = 64 to columns of its own.
    if constexpr (C::kRegSplit) setmaxnreg_dec<C::kRegKeyRow>();
    const int half = warp >= 12 ? 1 : 0;
    const int c0 = half * 64;  // first query of this warpgroup's half
    const int r = static_cast<int>((warp & 3) * 32 + lane_id());  // key row within the block == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint8_t* ds_row = smem + C::kOffDS + half * C::kBlockBytes + r * 128;
    const uint32_t swz = static_cast<uint32_t>(r & 7);
    bool ok = true;
    QCursor cur{i_begin, qh0};
    for (int it = 0; it < n_it; ++it) {
      q_advance(cur, it);
      const int st = it & 1;
      ok = mbar_wait(&sh.ld_full[st], (it >> 1) & 1, &sh.abort, &g_err_bwd) &&
           mbar_wait(&sh.s_full, it & 1, &sh.abort, &g_err_bwd);
      if (!ok) break;
      tc_fence_after();
      const float* l2 = s_lse2 + st * 128 + c0;
      const float* dd = s_dvec + st * 128 + c0;
      const bool diag = causal && (cur.i == kb);
      // window: query q of this block and key r are out of reach when
      // (query - key) >= window, i.e. dq0 + q - r >= window
      const int dq0 = (cur.i - kb) * 128;
      const bool wblk = WIN && dq0 + 127 >= window;
      // P stays fp32 for dS and goes to TMEM as bf16 pairs for dV.
      float p[64];
      uint32_t pw[32];
      auto p_quad = [&](const uint32_t (&rr)[32], int cc, int i4, float (&pv)[4]) {
        const float4 lq = reinterpret_cast<const float4*>(l2)[cc * 8 + i4];  // -L log2 e, 4 queries
        const int i = i4 * 4;
        const float2 c2 = make_float2(scale_log2, scale_log2);
        const float2 x01 = __ffma2_rn(make_float2(__uint_as_float(rr[i]), __uint_as_float(rr[i + 1])), c2,
                                      make_float2(lq.x, lq.y));
        const float2 x23 = __ffma2_rn(make_float2(__uint_as_float(rr[i + 2]), __uint_as_float(rr[i + 3])), c2,
                                      make_float2(lq.z, lq.w));
        const float xv[4] = {ex2_approx(x01.x), ex2_approx(x01.y), ex2_approx(x23.x), ex2_approx(x23.y)};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int q = c0 + cc * 32 + i + u;
          if constexpr (WIN) pv[u] = ((diag && q < r) || (wblk && dq0 + q - r >= window)) ? 0.f : xv[u];
          else pv[u] = (diag && q < r) ? 0.f : xv[u];  // query before key: masked
        }
      };
      {
        // Both TMEM loads of S^T before one wait (tcgen05.wait::ld waits for
        // every outstanding load), P packed as it is made.
        uint32_t rs[2][32];
        tmem_ld32(tmem + lane_base + C::kTmS + c0, rs[0]);
        tmem_ld32(tmem + lane_base + C::kTmS + c0 + 32, rs[1]);
        tmem_ld_wait(rs[0]);
        tmem_ld_wait(rs[1]);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc)
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            float pv[4];
            p_quad(rs[cc], cc, i4, pv);
#pragma unroll
            for (int u = 0; u < 4; ++u) p[cc * 32 + i4 * 4 + u] = pv[u];
            pw[cc * 16 + 2 * i4] = pack_bf16x2(pv[0], pv[1]);
            pw[cc * 16 + 2 * i4 + 1] = pack_bf16x2(pv[2], pv[3]);
          }
      }
      // (P_(i-1) there has been read: S_i, whose completion was awaited, was
      // issued after dV_(i-1).)
      tmem_st32(tmem + lane_base + C::kTmP + half * (C::kOwnP ? 32 : 96), pw);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&sh.p_ready);
      // dS_i may overwrite dS_(i-1) once dK_(i-1) and dQ_(i-1) have read it.
      ok = mbar_wait(&sh.dp_full, it & 1, &sh.abort, &g_err_bwd);
      if (ok && it > 0) ok = mbar_wait(&sh.dq_full, (it - 1) & 1, &sh.abort, &g_err_bwd);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t rr[32];
        tmem_ld32(tmem + lane_base + C::kTmDP + c0 + cc * 32, rr);
        tmem_ld_wait(rr);
        if constexpr (C::kEarly) {
          if (cc == 1) {  // dP^T's columns may take dP_(i+1)
            tc_fence_before();
            mbar_arrive(&sh.dp_free);
          }
        }
        // 32 queries = four 16-byte chunks of 8 in this half's column block
        uint32_t w[16];
#pragma unroll
        for (int i2 = 0; i2 < 8; ++i2) {  // D for 4 queries per 16-byte broadcast load
          const float4 dq4 = reinterpret_cast<const float4*>(dd)[cc * 8 + i2];  // -D
          const int q0 = cc * 32 + 4 * i2;
          const float2 a = __fmul2_rn(make_float2(p[q0], p[q0 + 1]),
                                      __fadd2_rn(make_float2(__uint_as_float(rr[4 * i2]), __uint_as_float(rr[4 * i2 + 1])),
                                                 make_float2(dq4.x, dq4.y)));
          const float2 b = __fmul2_rn(make_float2(p[q0 + 2], p[q0 + 3]),
                                      __fadd2_rn(make_float2(__uint_as_float(rr[4 * i2 + 2]), __uint_as_float(rr[4 * i2 + 3])),
                                                 make_float2(dq4.z, dq4.w)));
          w[2 * i2] = pack_bf16x2(a.x, a.y);
          w[2 * i2 + 1] = pack_bf16x2(b.x, b.y);
        }
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4) {
          const uint32_t chunk = static_cast<uint32_t>(cc * 4 + c4);
          *reinterpret_cast<uint4*>(ds_row + ((chunk ^ swz) << 4)) =
              make_uint4(w[4 * c4], w[4 * c4 + 1], w[4 * c4 + 2], w[4 * c4 + 3]);
        }
      }
      fence_proxy_async_smem();  // generic-proxy stores -> tensor core reads
      tc_fence_before();
      mbar_arrive(&sh.ds_ready);
      mbar_arrive(&sh.ld_empty[st]);
    }
    // dV = sum_i P_i^T dO_i, each warpgroup writing half of the columns, staged
    // with the 128-byte swizzle in K's dead space (every product has completed
    // once acc_done has) and written by TMA stores, which drop rows past N
    // (measured against per-thread row stores: +4 % on the backward at N = 512
    // and 1024, d = 128).  At d = 128 each warpgroup's 64 columns are a box of
    // their own; at d = 64 the two halves share one box.
    if constexpr (SPLIT) {
      // This CTA's part of dV (fp32), its 32-column blocks staged with the
      // 128-byte swizzle (warpgroup 0 in K's dead space, 1 in Q's first
      // stage) and added into the K/V head's accumulator by TMA reduce-adds.
      constexpr int kCols = D / 2;
      bool ok2 = ok && mbar_wait(&sh.acc_done, 0, &sh.abort, &g_err_bwd);
      uint8_t* stage = smem + (half ? C::kOffQ : C::kOffK);
      if (ok2) {
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < kCols; cc += 32) {
          uint32_t rr[32];
          tmem_ld32(tmem + lane_base + C::kTmDV + half * kCols + cc, rr);
          tmem_ld_wait(rr);
          uint8_t* row = stage + (cc / 32) * C::kBlockBytes + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(row + ((static_cast<uint32_t>(c) ^ swz) << 4)) =
                make_uint4(rr[4 * c], rr[4 * c + 1], rr[4 * c + 2], rr[4 * c + 3]);
        }
        fence_proxy_async_smem();
      }
      ok2 = named_bar_and(2 + half, 128, ok2);
      if (ok2 && (warp & 3) == 0 && lane_id() == 0) {
#pragma unroll
        for (int cc = 0; cc < kCols; cc += 32)
          tma_reduce_add_3d(&map_dv, half * kCols + cc, kb * 128, bh, stage + (cc / 32) * C::kBlockBytes);
        bulk_commit_group();
        bulk_wait_read_all();
      }
    } else {
      constexpr int kCols = D / 2;
      bool ok2 = ok && mbar_wait(&sh.acc_done, 0, &sh.abort, &g_err_bwd);
      if (ok2) {
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < kCols; cc += 32) {
          const int col = half * kCols + cc;
          uint32_t rr[32];
          tmem_ld32(tmem + lane_base + C::kTmDV + col, rr);
          tmem_ld_wait(rr);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(__uint_as_float(rr[2 * i]), __uint_as_float(rr[2 * i + 1]));
          uint8_t* box = smem + C::kOffK + (col / 64) * C::kBlockBytes;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(box + r * 128 + ((static_cast<uint32_t>((col % 64) / 8 + i) ^ swz) << 4)) =
                make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
        fence_proxy_async_smem();
      }
      if constexpr (D == 128) {
        ok2 = named_bar_and(2 + half, 128, ok2);
        if (ok2 && (warp & 3) == 0 && lane_id() == 0) {
          tma_store_3d(&map_dv, half * 64, kb * 128, bh, smem + C::kOffK + half * C::kBlockBytes);
          bulk_commit_group();
          bulk_wait_read_all();
        }
      } else {
        ok2 = named_bar_and(2, 256, ok2);
        if (ok2 && threadIdx.x == 0) {
          tma_store_3d(&map_dv, 0, kb * 128, bh, smem + C::kOffK);
          bulk_commit_group();
          bulk_wait_read_all();
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dQ reduction (query rows), dK epilogue
    if constexpr (C::kRegSplit) setmaxnreg_inc<C::kRegDq>();
    // dQ_i goes TMEM -> registers -> swizzled staging in shared memory ->
    // TMA reduce-add into the fp32 accumulator (the tensor map clips rows past N).
    const int r = threadIdx.x - 128;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t swz = static_cast<uint32_t>(r & 7);
    uint8_t* stage_row = smem + C::kOffStage + r * 128;
    const bool leader = (threadIdx.x == 128);
    bool ok = true;
    bool staged_before = false;
    QCursor cur{i_begin, qh0};
    for (int it = 0; it < n_it; ++it) {
      q_advance(cur, it);
      ok = mbar_wait(&sh.dq_full, it & 1, &sh.abort, &g_err_bwd);
      if (!ok) break;
      tc_fence_after();
      float v[D];
      // At d = 128 all four loads go out before one wait (measured: -1.3 % backward
      // time on the long causal workload); at d = 64 one at a time.
      if constexpr (D == 128) {
        uint32_t rr[D / 32][32];
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) tmem_ld32(tmem + lane_base + C::kTmDQ + cc * 32, rr[cc]);
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) tmem_ld_wait(rr[cc]);
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc)
#pragma unroll
          for (int i = 0; i < 32; ++i) v[cc * 32 + i] = __uint_as_float(rr[cc][i]);
      } else {
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t rr[32];
          tmem_ld32(tmem + lane_base + C::kTmDQ + cc * 32, rr);
          tmem_ld_wait(rr);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[cc * 32 + i] = __uint_as_float(rr[i]);
        }
      }
      tc_fence_before();
      mbar_arrive(&sh.dq_free);
      const int qrow0 = cur.i * 128;
      const int qh = cur.h;
      // 32-column blocks (128 rows x 128 bytes, swizzled for the reduce-add)
      // alternate between the two halves of the staging buffer, so that the
      // rows of block b are written while block b-1 is still being read.
#pragma unroll
      for (int b = 0; b < D / 32; ++b) {
        if (staged_before || b >= 2) {
          if (leader) bulk_wait_read_1();  // the reduce from this half (two blocks back) has read it
          named_bar_sync(1, 128);
        }
        uint8_t* blk = stage_row + (b & 1) * C::kBlockBytes;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int col = b * 32 + c * 4;
          *reinterpret_cast<float4*>(blk + ((static_cast<uint32_t>(c) ^ swz) << 4)) =
              make_float4(v[col], v[col + 1], v[col + 2], v[col + 3]);
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (leader) {
          tma_reduce_add_3d(&map_dq, b * 32, qrow0, qh, smem + C::kOffStage + (b & 1) * C::kBlockBytes);
          bulk_commit_group();
        }
      }
      staged_before = true;
    }
    if (leader) bulk_wait_read_all();
    // dK = scale * sum_i dS_i^T Q_i, staged in V's dead space (D / 64 boxes of
    // 64 columns) and written by TMA stores; with SPLIT this CTA's part in
    // fp32 (32-column blocks in V's dead space, then Q's second stage), added
    // into the K/V head's accumulator by TMA reduce-adds.
    if constexpr (SPLIT) {
      constexpr int kInV = C::kTileBytes / C::kBlockBytes;  // blocks that fit in V's space
      auto blk = [&](int b) { return smem + (b < kInV ? C::kOffV + b * C::kBlockBytes
                                                       : C::kOffQ + C::kTileBytes + (b - kInV) * C::kBlockBytes); };
      bool ok2 = ok && mbar_wait(&sh.acc_done, 0, &sh.abort, &g_err_bwd);
      if (ok2) {
        tc_fence_after();
#pragma unroll
        for (int b = 0; b < D / 32; ++b) {
          uint32_t rr[32];
          tmem_ld32(tmem + lane_base + C::kTmDK + b * 32, rr);
          tmem_ld_wait(rr);
          uint8_t* row = blk(b) + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<float4*>(row + ((static_cast<uint32_t>(c) ^ swz) << 4)) =
                make_float4(__uint_as_float(rr[4 * c]) * scale, __uint_as_float(rr[4 * c + 1]) * scale,
                            __uint_as_float(rr[4 * c + 2]) * scale, __uint_as_float(rr[4 * c + 3]) * scale);
        }
        fence_proxy_async_smem();
      }
      ok2 = named_bar_and(1, 128, ok2);
      if (ok2 && leader) {
#pragma unroll
        for (int b = 0; b < D / 32; ++b) tma_reduce_add_3d(&map_dk, b * 32, kb * 128, bh, blk(b));
        bulk_commit_group();
        bulk_wait_read_all();
      }
    } else {
      bool ok2 = ok && mbar_wait(&sh.acc_done, 0, &sh.abort, &g_err_bwd);
      if (ok2) {
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t rr[32];
          tmem_ld32(tmem + lane_base + C::kTmDK + cc, rr);
          tmem_ld_wait(rr);
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            pk[i] = pack_bf16x2(__uint_as_float(rr[2 * i]) * scale, __uint_as_float(rr[2 * i + 1]) * scale);
          uint8_t* box = smem + C::kOffV + (cc / 64) * C::kBlockBytes;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            *reinterpret_cast<uint4*>(box + r * 128 + ((static_cast<uint32_t>((cc % 64) / 8 + i) ^ swz) << 4)) =
                make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
        fence_proxy_async_smem();
      }
      ok2 = named_bar_and(1, 128, ok2);
      if (ok2 && leader) {
#pragma unroll
        for (int b = 0; b < D / 64; ++b)
          tma_store_3d(&map_dk, b * 64, kb * 128, bh, smem + C::kOffV + b * C::kBlockBytes);
        bulk_commit_group();
        bulk_wait_read_all();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool WIN, bool SPLIT>
fa_status launch_bwd_main_impl(const BwdArgs& a, cudaStream_t stream) {
  using C = BwdCfg<D>;
  const int BHq = a.B * a.H;     // query heads
  const int BH = a.B * a.Hkv;    // key/value heads: one CTA column each (SPLIT: one per query head)
  const int qgroup = a.H / a.Hkv;
  CUtensorMap mq, mk, mv, mdo, mdq, mdk, mdv;
  // SPLIT: dk and dv are the fp32 accumulators, reduced into like dq_acc.
  const int kv_eb = SPLIT ? 4 : 2, kv_box = SPLIT ? 32 : 64;
  if (!encode_rows_map(&mq, a.q, 2, D, a.N, BHq, 64, 128) || !encode_rows_map(&mk, a.k, 2, D, a.N, BH, 64, 128) ||
      !encode_rows_map(&mv, a.v, 2, D, a.N, BH, 64, 128) || !encode_rows_map(&mdo, a.dO, 2, D, a.N, BHq, 64, 128) ||
      !encode_rows_map(&mdq, a.dq_acc, 4, D, a.N, BHq, 32, 128) ||
      !encode_rows_map(&mdk, a.dk, kv_eb, D, a.N, BH, kv_box, 128) ||
      !encode_rows_map(&mdv, a.dv, kv_eb, D, a.N, BH, kv_box, 128))
    return FA_ERR_LAUNCH;
  auto kern = fa_bwd_main_kernel<D, WIN, SPLIT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes) != cudaSuccess)
    return FA_ERR_LAUNCH;
  if (C::kRegSplit) {
    // The setmaxnreg shares assume the launch allocation; with any other
    // count the dQ warpgroup's increase could never be granted.
    cudaFuncAttributes fattr{};
    if (cudaFuncGetAttributes(&fattr, kern) != cudaSuccess) return FA_ERR_LAUNCH;
    if (fattr.numRegs != kRegLaunch) return FA_ERR_KERNEL_CONFIG;
  }
  const int n_blk = (a.N + 127) / 128;
  // Heads per group: Q, dO (bf16) and the dQ accumulator (fp32) of a group
  // should stay within about 48 MB of the L2.
  const int items = SPLIT ? BHq : BH;
  const long long head_bytes = static_cast<long long>(a.N) * D * (2 + 2 + 4) * (SPLIT ? 1 : qgroup);
  int group = static_cast<int>(std::max<long long>(1, (48ll << 20) / head_bytes));
  group = std::min(group, items);
  dim3 grid(static_cast<unsigned>(n_blk * items));
  const cudaError_t e = launch_pdl(kern, grid, dim3(kThreads), C::kSmemBytes, stream, mq, mk, mv, mdo, mdq, mdk, mdv,
                                   a.lse, a.D, items, a.N, a.causal, a.scale, a.scale * kLog2e, group, a.H, qgroup,
                                   a.window);
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

fa_status launch_bwd_preprocess(const void* o, const void* dO, float* D, float* dq_acc, long long rows, int d,
                                cudaStream_t stream) {
  const int rows_per_block = 256 / (d / 8);
  const long long blocks = (rows + rows_per_block - 1) / rows_per_block;
  if (blocks > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  // A plain launch except for small problems: launched early, its many small
  // CTAs sit beside the previous kernel's last CTAs and slow them (measured:
  // +4 % on the long causal step, +2 % at N = 512 and 1024 with B*H = 512 and
  // 256), while at B*H*N <= 65536 rows the overlap wins (it and the convert
  // launched early: the GPT-2-small-like fwd+bwd step 70.5 -> 65.5 us).  Either
  // way the backward main kernel may launch early behind it.
  const auto* o16 = static_cast<const __nv_bfloat16*>(o);
  const auto* do16 = static_cast<const __nv_bfloat16*>(dO);
  const dim3 grid(static_cast<unsigned>(blocks));
  cudaError_t e;
  if (rows <= kSmallRows) {
    e = d == 64 ? launch_pdl(fa_bwd_preprocess_kernel<64>, grid, dim3(256), 0, stream, o16, do16, D, dq_acc, rows)
                : launch_pdl(fa_bwd_preprocess_kernel<128>, grid, dim3(256), 0, stream, o16, do16, D, dq_acc, rows);
  } else {
    if (d == 64) fa_bwd_preprocess_kernel<64><<<grid, 256, 0, stream>>>(o16, do16, D, dq_acc, rows);
    else fa_bwd_preprocess_kernel<128><<<grid, 256, 0, stream>>>(o16, do16, D, dq_acc, rows);
    e = cudaPeekAtLastError();
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

fa_status launch_bwd_main(const BwdArgs& a, cudaStream_t stream) {
  if (a.window > 0)
    return a.d == 64 ? launch_bwd_main_impl<64, true, false>(a, stream) : launch_bwd_main_impl<128, true, false>(a, stream);
  if (a.split_heads)
    return a.d == 64 ? launch_bwd_main_impl<64, false, true>(a, stream) : launch_bwd_main_impl<128, false, true>(a, stream);
  return a.d == 64 ? launch_bwd_main_impl<64, false, false>(a, stream)
                   : launch_bwd_main_impl<128, false, false>(a, stream);
}

fa_status launch_bwd_dq_convert(const float* dq_acc, void* dq, long long rows, int d, float scale,
                                cudaStream_t stream) {
  const long long n8 = rows * d / 8;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (n8 + 255) / 256;
  const long long cap = static_cast<long long>(sms) * 8;  // grid-stride beyond 8 waves of 256 threads
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  // Launched as the preprocess kernel is: early only for small problems.
  cudaError_t e;
  if (rows <= kSmallRows) {
    e = launch_pdl(fa_bwd_dq_convert_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, dq_acc,
                   static_cast<__nv_bfloat16*>(dq), n8, scale);
  } else {
    fa_bwd_dq_convert_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(dq_acc,
                                                                                 static_cast<__nv_bfloat16*>(dq), n8, scale);
    e = cudaPeekAtLastError();
  }
  return e == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

uint32_t bwd_take_error(cudaStream_t s) {
  uint32_t v = 0, zero = 0;
  cudaMemcpyFromSymbolAsync(&v, g_err_bwd, sizeof(v), 0, cudaMemcpyDeviceToHost, s);
  cudaStreamSynchronize(s);
  cudaMemcpyToSymbolAsync(g_err_bwd, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
  cudaStreamSynchronize(s);
  return v;
}

}  // namespace fa
