// Decode attention for sm_103a: one query row per (batch, query head) against
// a long key/value cache, the step that generates one token ("FlashAttention
// 三代演进", the decode case -- batch of short queries, memory-bound, tiled
// differently from the forward over whole sequences; the row it computes is the
// standard attention of "FLASH-ATTN", FlashAttention-2 > Background).
//
// The work is reading K and V once, so the kernels are organised for HBM
// bandwidth.  With one query head per key/value head (below) the products
// are dot products and P.V on the FMA pipes; with 2..16 query heads sharing a
// key/value head they are small contractions over the group and run on the
// tensor cores (fa_decode_tc_kernel, further down).  The CUDA-core kernel:
//  * the keys of one key/value head are cut into chunks; one CTA takes one
//    chunk for all the query heads that share that key/value head (grouped
//    queries read the cache once), and enough chunks exist to fill the GPU;
//  * a TMA warp streams the chunk's K tiles, then its V tiles (64 keys each,
//    128-byte swizzle) through a 3-slot ring guarded by full/empty mbarriers;
//    three CTAs share an SM;
//  * pass 1: 4 threads per key compute the scaled scores q_h . k (in log2
//    units) of every query head, packed fp32x2 FMAs, into shared memory;
//  * per head, the chunk's maximum m and sum l of 2^(s - m), with s replaced
//    by p = 2^(s - m) in place;
//  * pass 2: each thread owns two output columns for a quarter of the keys and
//    accumulates sum p v for every head; the quarters are summed at the end;
//  * the chunk's (m, l, unnormalised O) go to a workspace, and a second kernel
//    merges the chunks of a row with the block-merge rule of "FLASH-ATTN",
//    FlashAttention > Tiling and Recomputation: m = max m_c,
//    l = sum l_c 2^(m_c - m), O = sum O_c 2^(m_c - m) / l, L = m ln 2 + ln l.
#include <cuda_bf16.h>

#include "fa_common.cuh"
#include "fa_host.h"

namespace fa {

namespace {

__device__ uint32_t g_err_dec;

constexpr int kDecCompute = 256;           // 8 compute warps
constexpr int kDecThreads = kDecCompute + 32;  // + the TMA warp
constexpr int kDecTile = 64;               // keys per K or V tile
constexpr int kDecSlots = 3;
constexpr int kDecScoreBytes = 16384;      // chunk keys x padded heads x 4 bytes

template <int D>
struct DecCfg {
  static constexpr int kColBlocks = D * 2 / 128;        // 128-byte column blocks of a row
  static constexpr int kBlockBytes = kDecTile * 128;    // one column block of a tile
  static constexpr int kTileBytes = kDecTile * D * 2;   // one K or V tile
  static constexpr int kQuarter = D / 4;                // elements of a row per score thread
  static constexpr int kQStride = kQuarter + 4;         // padded fp32 quarter row of q
  static constexpr int kPairs = D / 2;                  // column pairs (pass 2)
  static constexpr int kGroups = kDecCompute / kPairs;  // key groups (pass 2)
  static constexpr int kKeysPerGroup = kDecTile / kGroups;
  static_assert(D == 64 || D == 128, "head dim");
  // The ring also holds the key-group sums at the end ([kGroups][g][D] fp32).
  __host__ __device__ static constexpr int ring_bytes(int g4) {
    return kDecSlots * kTileBytes > kGroups * g4 * D * 4 ? kDecSlots * kTileBytes : kGroups * g4 * D * 4;
  }
};

struct DecSmem {
  uint64_t full[kDecSlots];
  uint64_t empty[kDecSlots];
  float m[16];
  float l[16];
  float red_m[8][16];  // per compute warp and head
  float red_l[8][16];
  CtaAbort abort;
};

// Byte offset of element (row r, column e) of a tile stored as column blocks of
// 64 rows x 128 bytes with the 128-byte swizzle (16-byte chunk c of row r at
// chunk c ^ (r & 7)).
__device__ __forceinline__ int swz_off(int r, int e) {
  const int cb = e >> 6;
  const int c = (e & 63) >> 3;
  return cb * (kDecTile * 128) + r * 128 + (((c ^ (r & 7)) << 4) | ((e & 7) << 1));
}

__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// grid (nsplit, B*Hkv); each CTA: keys [chunk*C, min(N, chunk*C + C)) of one
// key/value head, for its g query heads.  G: g fixed at compile time, or 16
// for any g up to 16 read at run time; launched for g = 1 (grouped heads go to
// the tensor-core kernel below, which measured faster from g = 2).
template <int D, int G>
__global__ void __launch_bounds__(kDecThreads, 3)
    fa_decode_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                     const __nv_bfloat16* __restrict__ q, float* __restrict__ part, int H, int Hkv, int N, int C,
                     int nsplit, float scale_log2) {
  using Cf = DecCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ DecSmem sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int G4 = (G + 3) & ~3;
  uint8_t* s_ring = smem;                                         // kDecSlots tiles
  float* s_score = reinterpret_cast<float*>(smem + Cf::ring_bytes(G4));  // [C][gp]
  float* s_q = s_score + kDecScoreBytes / 4;                      // [g][4][kQStride]

  if (*reinterpret_cast<volatile uint32_t*>(&g_err_dec) & FA_DEVERR_TIMEOUT) return;
  const int g = G < 16 ? G : H / Hkv;
  const int gp = (g + 3) & ~3;
  const int chunk = static_cast<int>(blockIdx.x);
  const int bkv = static_cast<int>(blockIdx.y);  // b * Hkv + kv head
  const int key_begin = chunk * C;
  const int key_end = min(N, key_begin + C);
  const int n_tiles = (key_end - key_begin + kDecTile - 1) / kDecTile;
  const int bq0 = (bkv / Hkv) * H + (bkv % Hkv) * g;  // first query row (b * H + h)
  const int warp = static_cast<int>(warp_id());

  if (threadIdx.x == 0) {
    sh.abort.flag = 0;
    for (int s = 0; s < kDecSlots; ++s) {
      mbar_init(&sh.full[s], 1);
      mbar_init(&sh.empty[s], kDecCompute / 32);
    }
    fence_barrier_init();
  }
  // Set-up done: the next kernel may start launching; q, the cache and the
  // workspace are touched only after the kernels before this one completed.
  pdl_launch_dependents();
  pdl_wait_prior();
  // q of the group, fp32, times scale * log2 e, each quarter row padded so that
  // the four quarters fall in different banks.
  for (int i = threadIdx.x; i < g * D; i += kDecThreads) {
    const int h = i / D, e = i % D;
    s_q[(h * 4 + e / Cf::kQuarter) * Cf::kQStride + e % Cf::kQuarter] =
        __bfloat162float(q[static_cast<size_t>(bq0 + h) * D + e]) * scale_log2;
  }
  __syncthreads();

  if (warp == kDecCompute / 32) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      int issued = 0;
      for (int it = 0; it < 2 * n_tiles && !sh.abort.flag; ++it) {
        const int slot = issued % kDecSlots;
        const int round = issued / kDecSlots;
        if (round > 0 && !mbar_wait<true>(&sh.empty[slot], (round - 1) & 1, &sh.abort, &g_err_dec)) break;
        const bool is_k = it < n_tiles;
        const int key0 = key_begin + (is_k ? it : it - n_tiles) * kDecTile;
        mbar_arrive_expect_tx(&sh.full[slot], Cf::kTileBytes);
        for (int cb = 0; cb < Cf::kColBlocks; ++cb)
          tma_load_3d(s_ring + slot * Cf::kTileBytes + cb * Cf::kBlockBytes, is_k ? &map_k : &map_v, cb * 64, key0,
                      bkv, &sh.full[slot]);
        ++issued;
      }
      if (sh.abort.flag) {
        for (int s = 0; s < kDecSlots && s < issued; ++s) {
          const int last = s + ((issued - 1 - s) / kDecSlots) * kDecSlots;
          mbar_wait_drain(&sh.full[s], (last / kDecSlots) & 1, &g_err_dec);
        }
      }
    }
    __syncwarp();
    return;
  }

  // ---------------------------------------------------------------- compute
  const int t = threadIdx.x;
  bool ok = true;
  int used = 0;  // ring uses so far
  auto acquire = [&](int slot) {  // warp-uniform result: the warp shuffles after it
    const bool got = ok && mbar_wait<true>(&sh.full[slot], (used / kDecSlots) & 1, &sh.abort, &g_err_dec);
    ok = __all_sync(0xffffffffu, got);
    return ok;
  };
  auto release = [&](int slot) {
    __syncwarp();
    if (lane_id() == 0) mbar_arrive(&sh.empty[slot]);
    ++used;
  };

  // Pass 1: scores.  Thread t: key k = t / 4 of the tile, quarter p = t % 4.
  // Each thread also keeps the running maximum of the heads it stores
  // (h % 4 == p).
  float mloc[G4 / 4];
#pragma unroll
  for (int i = 0; i < G4 / 4; ++i) mloc[i] = -INFINITY;
  {
    const int k = t >> 2, p = t & 3;
    const float* qp = s_q + p * Cf::kQStride;
    for (int tile = 0; tile < n_tiles; ++tile) {
      const int slot = used % kDecSlots;
      if (!acquire(slot)) break;
      const uint8_t* kt = s_ring + slot * Cf::kTileBytes;
      float2 acc[G];
#pragma unroll
      for (int h = 0; h < G; ++h) acc[h] = make_float2(0.f, 0.f);
#pragma unroll
      for (int c = 0; c < Cf::kQuarter / 8; ++c) {  // 16-byte chunks of the quarter
        const uint4 w = *reinterpret_cast<const uint4*>(kt + swz_off(k, p * Cf::kQuarter + c * 8));
        const float2 k0 = bf16x2_to_float2(w.x), k1 = bf16x2_to_float2(w.y);
        const float2 k2 = bf16x2_to_float2(w.z), k3 = bf16x2_to_float2(w.w);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          if (h < g) {
            const float4 qa = *reinterpret_cast<const float4*>(qp + h * 4 * Cf::kQStride + c * 8);
            const float4 qb = *reinterpret_cast<const float4*>(qp + h * 4 * Cf::kQStride + c * 8 + 4);
            acc[h] = __ffma2_rn(k0, make_float2(qa.x, qa.y), acc[h]);
            acc[h] = __ffma2_rn(k1, make_float2(qa.z, qa.w), acc[h]);
            acc[h] = __ffma2_rn(k2, make_float2(qb.x, qb.y), acc[h]);
            acc[h] = __ffma2_rn(k3, make_float2(qb.z, qb.w), acc[h]);
          }
        }
      }
      release(slot);
      const int key = tile * kDecTile + k;  // within the chunk
      const bool valid = key_begin + key < key_end;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        if (h < g) {
          float v = acc[h].x + acc[h].y;
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          if ((h & 3) == p) {
            s_score[key * gp + h] = valid ? v : -INFINITY;
            if (valid) mloc[h >> 2] = fmaxf(mloc[h >> 2], v);
          }
        }
      }
    }
  }
  // Per head: m = max over the chunk (from the threads' running maxima),
  // p = 2^(s - m) in place over all threads, l = sum p.
  {
    const int p = t & 3;
#pragma unroll
    for (int i = 0; i < G4 / 4; ++i) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1)  // lanes of the same p
        mloc[i] = fmaxf(mloc[i], __shfl_xor_sync(0xffffffffu, mloc[i], off));
      if (lane_id() < 4) sh.red_m[warp][4 * i + p] = mloc[i];
    }
  }
  named_bar_sync(1, kDecCompute);
  float m[G4], l[G4];
#pragma unroll
  for (int h = 0; h < G4; ++h) {
    float mm = sh.red_m[0][h];
#pragma unroll
    for (int w = 1; w < kDecCompute / 32; ++w) mm = fmaxf(mm, sh.red_m[w][h]);
    m[h] = mm == -INFINITY ? 0.0f : mm;  // padded heads: no keys
    l[h] = 0.f;
  }
  const int n_keys = n_tiles * kDecTile;
  for (int key = t; key < n_keys; key += kDecCompute) {
#pragma unroll
    for (int h4 = 0; h4 < G4; h4 += 4) {
      if (h4 < gp) {
        float4 s4 = *reinterpret_cast<const float4*>(s_score + key * gp + h4);
        s4.x = ex2_approx(s4.x - m[h4]);
        s4.y = ex2_approx(s4.y - m[h4 + 1]);
        s4.z = ex2_approx(s4.z - m[h4 + 2]);
        s4.w = ex2_approx(s4.w - m[h4 + 3]);
        *reinterpret_cast<float4*>(s_score + key * gp + h4) = s4;
        l[h4] += s4.x;
        l[h4 + 1] += s4.y;
        l[h4 + 2] += s4.z;
        l[h4 + 3] += s4.w;
      }
    }
  }
#pragma unroll
  for (int h = 0; h < G4; ++h) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
    if (lane_id() == 0) sh.red_l[warp][h] = l[h];
  }
  named_bar_sync(1, kDecCompute);
  if (t == 0) {  // unrolled over heads: m stays in registers
#pragma unroll
    for (int h = 0; h < G4; ++h) {
      if (h < g) {
        float ls = 0.f;
#pragma unroll
        for (int w = 0; w < kDecCompute / 32; ++w) ls += sh.red_l[w][h];
        sh.m[h] = m[h];
        sh.l[h] = ls;
      }
    }
  }

  // Pass 2: O_h += sum_k p_hk v_k.  Thread t: column pair cp, key group kg.
  const int cp = t % Cf::kPairs, kg = t / Cf::kPairs;
  float2 o[G4];
#pragma unroll
  for (int h = 0; h < G4; ++h) o[h] = make_float2(0.f, 0.f);
  for (int tile = 0; tile < n_tiles; ++tile) {
    const int slot = used % kDecSlots;
    if (!acquire(slot)) break;
    const uint8_t* vt = s_ring + slot * Cf::kTileBytes;
#pragma unroll
    for (int kk = 0; kk < Cf::kKeysPerGroup; ++kk) {
      const int k = kg * Cf::kKeysPerGroup + kk;
      const float2 v = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(vt + swz_off(k, 2 * cp)));
      const float* pk = s_score + (tile * kDecTile + k) * gp;
#pragma unroll
      for (int h4 = 0; h4 < G4; h4 += 4) {
        if (h4 < g) {
          const float4 p4 = *reinterpret_cast<const float4*>(pk + h4);
          o[h4] = __ffma2_rn(make_float2(p4.x, p4.x), v, o[h4]);
          o[h4 + 1] = __ffma2_rn(make_float2(p4.y, p4.y), v, o[h4 + 1]);
          o[h4 + 2] = __ffma2_rn(make_float2(p4.z, p4.z), v, o[h4 + 2]);
          o[h4 + 3] = __ffma2_rn(make_float2(p4.w, p4.w), v, o[h4 + 3]);
        }
      }
    }
    release(slot);
  }
  // Sum the key groups through shared memory: past this barrier every issued
  // copy has been consumed, so the ring is free.
  const bool all_ok = named_bar_and(1, kDecCompute, ok);
  float* red = reinterpret_cast<float*>(s_ring);  // [kGroups][g][D]
#pragma unroll
  for (int h = 0; h < G4; ++h)  // unrolled: o stays in registers
    if (h < g) *reinterpret_cast<float2*>(red + (kg * g + h) * D + 2 * cp) = o[h];
  named_bar_sync(1, kDecCompute);
  if (all_ok) {
    const size_t stride = D + 4;
    for (int i = t; i < g * D; i += kDecCompute) {
      const int h = i / D, e = i % D;
      float s = 0.f;
#pragma unroll
      for (int gg = 0; gg < Cf::kGroups; ++gg) s += red[(gg * g + h) * D + e];
      float* row = part + (static_cast<size_t>(bq0 + h) * nsplit + chunk) * stride;
      row[e] = s;
      if (e == 0) {
        row[D] = sh.m[h];
        row[D + 1] = sh.l[h];
      }
    }
  }
}

// One warp per query row: merge its nsplit chunks.
template <int D>
__global__ void __launch_bounds__(256) fa_decode_merge_kernel(const float* __restrict__ part,
                                                              __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                              int rows, int nsplit) {
  constexpr int E = D / 32;
  pdl_launch_dependents();
  pdl_wait_prior();  // the chunks' partials come from the kernel before
  const int row = static_cast<int>(blockIdx.x) * 8 + static_cast<int>(warp_id());
  if (row >= rows) return;
  const size_t stride = D + 4;
  const float* base = part + static_cast<size_t>(row) * nsplit * stride;
  float m = -INFINITY;
  for (int s = 0; s < nsplit; ++s) m = fmaxf(m, base[s * stride + D]);
  float l = 0.f, acc[E];
#pragma unroll
  for (int j = 0; j < E; ++j) acc[j] = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float* r = base + s * stride;
    const float w = ex2_approx(r[D] - m);
    l += r[D + 1] * w;
#pragma unroll
    for (int j = 0; j < E; ++j) acc[j] += r[lane_id() * E + j] * w;
  }
  const float inv = 1.0f / l;
#pragma unroll
  for (int j = 0; j < E; ++j) o[static_cast<size_t>(row) * D + lane_id() * E + j] = __float2bfloat16_rn(acc[j] * inv);
  if (lane_id() == 0) lse[row] = m * 0.69314718055994531f + logf(l);
}

// Both decode kernels and the merge are launched with programmatic stream
// serialization: each signals its dependents after its set-up and waits for
// the kernels before it only where it first touches memory, so the merge's
// launch overlaps the decode kernel's last CTAs and the next call's set-up
// overlaps the merge.
template <int D>
fa_status launch_merge(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t s) {
  const int rows = a.B * a.H;
  return launch_pdl(fa_decode_merge_kernel<D>, dim3((rows + 7) / 8), dim3(256), 0, s, a.part,
                    static_cast<__nv_bfloat16*>(a.o), a.lse, rows, pl.nsplit) == cudaSuccess
             ? FA_OK
             : FA_ERR_LAUNCH;
}

template <int D, int G>
fa_status launch_decode_impl(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t s) {
  using Cf = DecCfg<D>;
  CUtensorMap mk, mv;
  const int BHkv = a.B * a.Hkv;
  if (!encode_rows_map(&mk, a.k, 2, D, a.N, BHkv, 64, kDecTile) ||
      !encode_rows_map(&mv, a.v, 2, D, a.N, BHkv, 64, kDecTile))
    return FA_ERR_LAUNCH;
  const int g = a.H / a.Hkv;
  const int smem = 1024 + Cf::ring_bytes((G + 3) & ~3) + kDecScoreBytes + g * 4 * Cf::kQStride * 4;
  auto kern = fa_decode_kernel<D, G>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
    return FA_ERR_LAUNCH;
  const dim3 grid(static_cast<unsigned>(pl.nsplit), static_cast<unsigned>(BHkv));
  if (launch_pdl(kern, grid, dim3(kDecThreads), smem, s, mk, mv, static_cast<const __nv_bfloat16*>(a.q), a.part, a.H,
                 a.Hkv, a.N, pl.chunk, pl.nsplit, a.scale * 1.4426950408889634f) != cudaSuccess)
    return FA_ERR_LAUNCH;
  return launch_merge<D>(a, pl, s);
}


// ---------------------------------------------------------------------------
// Grouped heads (2..16 query heads per key/value head): the score and
// P.V products are real contractions over the group, (keys x d)(d x heads)
// and (d x keys)(keys x heads), so they go to the tensor cores, which leaves
// the kernel bound by the cache read again.  A chunk's tiles are processed
// one at a time with the online softmax of "FLASH-ATTN", FlashAttention-2
// (per head a running maximum, raised only past a threshold, and a running
// sum), so K and V tiles stream interleaved and a chunk may be any length.
//   warps 0-3 : one key of a 128-key tile per thread (TMEM lane): per tile
//               the per-head maximum over the tile's keys, then P into shared
//               memory as the B operand of P.V; thread t also owns row d = t
//               of O^T, which it rescales when a head's maximum is raised,
//               and reads out at the end.
//   warp 4    : TMA producer: K_0, K_1, V_0, K_2, V_1, ... through a 3-slot
//               ring (the next tile's scores are computed during this one's
//               softmax).
//   warp 5    : TMEM allocation and the MMA-issuing thread.
// S^T = K Q^T (M = 128 keys, N = 16 padded heads, A = K tile K-major, B = Q
// K-major) in TMEM columns 16 (t & 1); O^T += V^T P^T (M = 128 rows of d,
// N = 16, A = V tile read MN-major, B = P K-major) in columns 128.. .  At
// d = 64 a ring slot keeps its 128-row size: the product's rows 64..127 read
// the slot's unused second half and are never read back.
constexpr int kTcThreads = 192;
constexpr int kTcTile = 128;           // keys per tile
constexpr int kTcSlots = 3;
constexpr int kTcTileBytes = kTcTile * 128 * 2;  // 32 KB: a 128-key tile at d = 128 (slot size)
constexpr int kTcBlockBytes = kTcTile * 128;     // one 64-column block of a tile
constexpr int kTcN = 16;               // padded heads
constexpr int kTcPBytes = kTcN * kTcTile * 2;    // 4 KB: P of one tile (16 x 128 bf16)
constexpr int kTcQBytes = kTcN * 128 * 2;        // 4 KB
constexpr uint32_t kTcTmO = 128;
constexpr float kTcTauLog2 = 8.0f;     // P <= 2^8 between raises of a head's maximum
constexpr int kTcSmem = 1024 + kTcSlots * kTcTileBytes + 2 * kTcPBytes + kTcQBytes;

struct DecTcSmem {
  uint64_t full[kTcSlots];
  uint64_t empty[kTcSlots];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t p_empty[2];
  uint64_t pv_done;
  uint64_t o_done;
  uint64_t drain;
  uint32_t tmem_base;
  float red[2][4][kTcN];   // per-tile maxima of the four warps (double-buffered by tile)
  float lred[4][kTcN];     // the warps' row sums at the end
  float m[kTcN];
  float l[kTcN];
  CtaAbort abort;
};

// Named barrier that also returns the OR of `v` over the participating threads.
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pin, pout;\n setp.ne.u32 pin, %1, 0;\n"
      " barrier.cta.red.or.pred pout, %2, %3, pin;\n selp.u32 %0, 1, 0, pout;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Byte offset of (row r, element e) in a K-major tile of `rows` rows stored as
// 64-element (128-byte) column blocks with the 128-byte swizzle.
__device__ __forceinline__ int kmaj_off(int r, int e, int rows) {
  return (e >> 6) * rows * 128 + r * 128 + ((((e & 63) >> 3) ^ (r & 7)) << 4) + ((e & 7) << 1);
}

// Ring order of a chunk's n tiles: K_0, then for each tile t, K_(t+1) (if
// any) and V_t.  Position of K_t and V_t in that order:
__device__ __forceinline__ int tc_k_pos(int t) { return t == 0 ? 0 : 2 * t - 1; }
__device__ __forceinline__ int tc_v_pos(int t, int n) { return t < n - 1 ? 2 * t + 2 : 2 * t + 1; }

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    fa_decode_tc_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                        const __nv_bfloat16* __restrict__ q, float* __restrict__ part, int H, int Hkv, int N, int C,
                        int nsplit, float scale_log2) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ DecTcSmem sh;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* s_ring = smem;
  uint8_t* s_p = smem + kTcSlots * kTcTileBytes;  // two P buffers
  uint8_t* s_qp = s_p + 2 * kTcPBytes;             // padded Q

  if (*reinterpret_cast<volatile uint32_t*>(&g_err_dec) & FA_DEVERR_TIMEOUT) return;
  const int g = H / Hkv;
  const int chunk = static_cast<int>(blockIdx.x);
  const int bkv = static_cast<int>(blockIdx.y);
  const int key_begin = chunk * C;
  const int key_end = min(N, key_begin + C);
  const int n_tiles = (key_end - key_begin + kTcTile - 1) / kTcTile;
  const int bq0 = (bkv / Hkv) * H + (bkv % Hkv) * g;
  const int warp = static_cast<int>(warp_id());
  const int t = threadIdx.x;

  if (t == 0) {
    sh.abort.flag = 0;
    for (int i = 0; i < kTcSlots; ++i) {
      mbar_init(&sh.full[i], 1);
      mbar_init(&sh.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sh.s_full[i], 1);
      mbar_init(&sh.p_full[i], 128);
      mbar_init(&sh.p_empty[i], 1);
    }
    mbar_init(&sh.pv_done, 1);
    mbar_init(&sh.o_done, 1);
    mbar_init(&sh.drain, 1);
    fence_barrier_init();
  }
  if (warp == 5) tmem_alloc(&sh.tmem_base, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh.tmem_base;
  // Set-up done: the next kernel may start launching; q, the cache and the
  // workspace are touched only after the kernels before this one completed.
  pdl_launch_dependents();
  pdl_wait_prior();
  // Q of the group as a 16-row K-major bf16 tile (rows past g are zero).
  for (int i = t; i < kTcN * D; i += kTcThreads) {
    const int h = i / D, e = i % D;
    const __nv_bfloat16 val = h < g ? q[static_cast<size_t>(bq0 + h) * D + e] : __float2bfloat16_rn(0.f);
    *reinterpret_cast<__nv_bfloat16*>(s_qp + kmaj_off(h, e, kTcN)) = val;
  }
  fence_proxy_async_smem();  // generic-proxy stores -> tensor core reads
  __syncthreads();

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (elect_one()) {
      tma_prefetch_desc(&map_k);
      tma_prefetch_desc(&map_v);
      int issued = 0;
      for (int i = 0; i < 2 * n_tiles && !sh.abort.flag; ++i) {
        const int slot = issued % kTcSlots;
        const int round = issued / kTcSlots;
        if (round > 0 && !mbar_wait<true>(&sh.empty[slot], (round - 1) & 1, &sh.abort, &g_err_dec)) break;
        // position i -> (K or V, tile), the inverse of tc_k_pos / tc_v_pos
        const bool is_k = i == 0 || (i != 2 * n_tiles - 1 && (i & 1));
        const int tile = i == 0 ? 0 : (i == 2 * n_tiles - 1 ? n_tiles - 1 : (is_k ? (i + 1) / 2 : (i - 2) / 2));
        const int key0 = key_begin + tile * kTcTile;
        mbar_arrive_expect_tx(&sh.full[slot], kTcTile * D * 2);
        for (int cb = 0; cb < D / 64; ++cb)
          tma_load_3d(s_ring + slot * kTcTileBytes + cb * kTcBlockBytes, is_k ? &map_k : &map_v, cb * 64, key0, bkv,
                      &sh.full[slot]);
        ++issued;
      }
      if (sh.abort.flag) {
        for (int i = 0; i < kTcSlots && i < issued; ++i) {
          const int last = i + ((issued - 1 - i) / kTcSlots) * kTcSlots;
          mbar_wait_drain(&sh.full[i], (last / kTcSlots) & 1, &g_err_dec);
        }
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (elect_one()) {
      constexpr uint32_t kIdS = idesc_bf16(128, kTcN, false, false);
      constexpr uint32_t kIdPV = idesc_bf16(128, kTcN, true, false);
      const uint64_t ring_k = sdesc_sw128(smem_u32(s_ring), 16, 1024);             // K tiles, K-major
      const uint64_t ring_mn = sdesc_sw128(smem_u32(s_ring), kTcBlockBytes, 1024);  // V tiles, MN-major
      const uint64_t q_k = sdesc_sw128(smem_u32(s_qp), 16, 1024);
      const uint64_t p_k = sdesc_sw128(smem_u32(s_p), 16, 1024);
      bool ok = true;
      // S^T of tile u into columns 16 (u & 1); the ring is consumed in order.
      auto issue_s = [&](int u) {
        const int pos = tc_k_pos(u);
        const int slot = pos % kTcSlots;
        ok = mbar_wait<true>(&sh.full[slot], (pos / kTcSlots) & 1, &sh.abort, &g_err_dec);
        if (!ok) return;
        tc_fence_after();
        const uint64_t a0 = sdesc_advance(ring_k, slot * kTcTileBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          mma_bf16_ss(tmem + (u & 1) * kTcN, sdesc_advance(a0, (kk >> 2) * kTcBlockBytes + (kk & 3) * 32),
                      sdesc_advance(q_k, (kk >> 2) * (kTcN * 128) + (kk & 3) * 32), kIdS, kk > 0);
        }
        tc_commit(&sh.s_full[u & 1]);
        tc_commit(&sh.empty[slot]);
      };
      issue_s(0);
      if (ok && n_tiles > 1) issue_s(1);
      for (int u = 0; ok && u < n_tiles; ++u) {
        const int b = u & 1;
        const int pos = tc_v_pos(u, n_tiles);
        const int slot = pos % kTcSlots;
        // P_u written (and S^T_u read) by the key warps, V_u landed
        ok = mbar_wait<true>(&sh.p_full[b], (u >> 1) & 1, &sh.abort, &g_err_dec) &&
             mbar_wait<true>(&sh.full[slot], (pos / kTcSlots) & 1, &sh.abort, &g_err_dec);
        if (!ok) break;
        tc_fence_after();
        const uint64_t a0 = sdesc_advance(ring_mn, slot * kTcTileBytes);
        const uint64_t b0 = sdesc_advance(p_k, b * kTcPBytes);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          mma_bf16_ss(tmem + kTcTmO, sdesc_advance(a0, kk * 2048),
                      sdesc_advance(b0, (kk >> 2) * (kTcN * 128) + (kk & 3) * 32), kIdPV, (u > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(&sh.p_empty[b]);
        tc_commit(&sh.empty[slot]);
        tc_commit(&sh.pv_done);
        if (u + 2 < n_tiles) issue_s(u + 2);  // into the columns S^T_u has left
      }
      if (ok) tc_commit(&sh.o_done);
      tc_commit(&sh.drain);
      mbar_wait_drain(&sh.drain, 0, &g_err_dec);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ keys (lanes)
    // Every thread takes every named barrier below; a failed wait only clears
    // `ok`, and the barriers that combine `ok` make all four warps stop
    // together.
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    bool ok = true;
    float m[kTcN], l[kTcN];  // per head: reference maximum (log2 units), this thread's partial sum
#pragma unroll
    for (int h = 0; h < kTcN; ++h) {
      m[h] = 0.f;
      l[h] = 0.f;
    }
    for (int u = 0; u < n_tiles; ++u) {
      const int b = u & 1;
      const bool valid = key_begin + u * kTcTile + t < key_end;
      float x[kTcN];
      ok = ok && mbar_wait<true>(&sh.s_full[b], (u >> 1) & 1, &sh.abort, &g_err_dec);
      if (ok) {
        tc_fence_after();
        uint32_t r[16];
        tmem_ld16(tmem + lane_base + b * kTcN, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int h = 0; h < kTcN; ++h) x[h] = valid ? __uint_as_float(r[h]) * scale_log2 : -INFINITY;
      } else {
#pragma unroll
        for (int h = 0; h < kTcN; ++h) x[h] = -INFINITY;
      }
      // Only a tile in which some key exceeds a head's reference by more than
      // the threshold (and the first tile) needs the tile's maxima: one
      // barrier tells every thread whether any did (a failed wait counts, so
      // that the barrier below combines the status).
      bool mine = u == 0 || !ok;
#pragma unroll
      for (int h = 0; h < kTcN; ++h) mine |= x[h] > m[h] + kTcTauLog2;
      const bool need = named_bar_or(1, 128, mine);
      bool raise = false;
      float alpha[kTcN];
#pragma unroll
      for (int h = 0; h < kTcN; ++h) alpha[h] = 1.0f;
      if (need) {
        // the tile's maximum per head over its 128 keys: warp, then the four warps
        float mt[kTcN];
#pragma unroll
        for (int h = 0; h < kTcN; ++h) {
          mt[h] = x[h];
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], off));
        }
        if (lane_id() == 0) {
#pragma unroll
          for (int h = 0; h < kTcN; ++h) sh.red[b][warp][h] = mt[h];
        }
        // (sh.red[b] is written again at a later tile, after every thread has
        // passed the next tile's barrier, so after this tile's reads)
        ok = named_bar_and(1, 128, ok);
        if (!ok) break;
#pragma unroll
        for (int h = 0; h < kTcN; ++h) {
          const float mm = fmaxf(fmaxf(sh.red[b][0][h], sh.red[b][1][h]), fmaxf(sh.red[b][2][h], sh.red[b][3][h]));
          if (u == 0) {
            m[h] = mm == -INFINITY ? 0.0f : mm;  // padded heads (and no visible key) use 0
          } else if (mm > m[h] + kTcTauLog2) {
            alpha[h] = ex2_approx(m[h] - mm);
            m[h] = mm;
            raise = true;
          }
        }
      }
      // (the same values in every thread: `raise` is uniform)
      if (raise) {
        // O^T is complete up to PV_(u-1); thread t rescales its row d = t
        ok = mbar_wait<true>(&sh.pv_done, (u - 1) & 1, &sh.abort, &g_err_dec);
        if (ok) {
          tc_fence_after();
          uint32_t r[16];
          tmem_ld16(tmem + lane_base + kTcTmO, r);
          tmem_ld_wait(r);
#pragma unroll
          for (int h = 0; h < kTcN; ++h) r[h] = __float_as_uint(__uint_as_float(r[h]) * alpha[h]);
          tmem_st16(tmem + lane_base + kTcTmO, r);
          tmem_st_wait();
        }
#pragma unroll
        for (int h = 0; h < kTcN; ++h) l[h] *= alpha[h];
      }
      if (ok && u >= 2)  // the P.V two tiles back has read this buffer
        ok = mbar_wait<true>(&sh.p_empty[b], ((u >> 1) - 1) & 1, &sh.abort, &g_err_dec);
      uint8_t* pb = s_p + b * kTcPBytes;
#pragma unroll
      for (int h = 0; h < kTcN; ++h) {
        const float pv = valid ? ex2_approx(x[h] - m[h]) : 0.f;
        l[h] += pv;
        if (ok) *reinterpret_cast<__nv_bfloat16*>(pb + kmaj_off(h, t, kTcN)) = __float2bfloat16_rn(pv);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&sh.p_full[b]);
    }
#pragma unroll
    for (int h = 0; h < kTcN; ++h) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) l[h] += __shfl_xor_sync(0xffffffffu, l[h], off);
    }
    if (lane_id() == 0) {
#pragma unroll
      for (int h = 0; h < kTcN; ++h) sh.lred[warp][h] = l[h];
    }
    const bool all_ok = named_bar_and(1, 128, ok);
    if (t == 0) {
#pragma unroll
      for (int h = 0; h < kTcN; ++h) {
        sh.m[h] = m[h];
        sh.l[h] = (sh.lred[0][h] + sh.lred[1][h]) + (sh.lred[2][h] + sh.lred[3][h]);
      }
    }
    named_bar_sync(1, 128);
    if (all_ok && mbar_wait<true>(&sh.o_done, 0, &sh.abort, &g_err_dec)) {
      tc_fence_after();
      uint32_t r[16];
      tmem_ld16(tmem + lane_base + kTcTmO, r);  // thread t: column d = t of O^T
      tmem_ld_wait(r);
      const size_t stride = D + 4;
#pragma unroll
      for (int h = 0; h < kTcN; ++h) {
        if (h < g && t < D) {
          float* row = part + (static_cast<size_t>(bq0 + h) * nsplit + chunk) * stride;
          row[t] = __uint_as_float(r[h]);
          if (t == 0) {
            row[D] = sh.m[h];
            row[D + 1] = sh.l[h];
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

template <int D>
fa_status launch_decode_tc_impl(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t s) {
  CUtensorMap mk, mv;
  const int BHkv = a.B * a.Hkv;
  if (!encode_rows_map(&mk, a.k, 2, D, a.N, BHkv, 64, kTcTile) ||
      !encode_rows_map(&mv, a.v, 2, D, a.N, BHkv, 64, kTcTile))
    return FA_ERR_LAUNCH;
  auto kern = fa_decode_tc_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem) != cudaSuccess)
    return FA_ERR_LAUNCH;
  const dim3 grid(static_cast<unsigned>(pl.nsplit), static_cast<unsigned>(BHkv));
  if (launch_pdl(kern, grid, dim3(kTcThreads), kTcSmem, s, mk, mv, static_cast<const __nv_bfloat16*>(a.q), a.part,
                 a.H, a.Hkv, a.N, pl.chunk, pl.nsplit, a.scale * 1.4426950408889634f) != cudaSuccess)
    return FA_ERR_LAUNCH;
  return launch_merge<D>(a, pl, s);
}

fa_status launch_decode_tc(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t s) {
  return a.d == 64 ? launch_decode_tc_impl<64>(a, pl, s) : launch_decode_tc_impl<128>(a, pl, s);
}

bool use_tc(int g, int d) { return g >= 2 && (d == 64 || d == 128); }

}  // namespace

DecodePlan decode_plan(int B, int H, int Hkv, int N, int d) {
  const int g = H / Hkv;
  const int gp = (g + 3) & ~3;
  const bool tc = use_tc(g, d);
  const long long units = static_cast<long long>(B) * Hkv;
  if (tc) {
    // Any chunk length (one tile at a time): one resident wave of at most two
    // CTAs per SM on 152 SMs, each streaming one chunk; past one wave, the
    // split of each (batch, key/value head) with the fewest waves per unit of
    // work.
    constexpr long long kWave = 2 * 152;
    const long long tiles = (N + kTcTile - 1) / kTcTile;
    long long ns = 1;
    if (units < kWave) {
      ns = kWave / units;
    } else {
      double best = 1e30;
      for (long long c = 1; c <= 4; ++c) {
        const double cost = static_cast<double>((units * c + kWave - 1) / kWave) / static_cast<double>(c);
        if (cost < best - 1e-9) {
          best = cost;
          ns = c;
        }
      }
    }
    if (ns > tiles) ns = tiles;
    if (ns < 1) ns = 1;
    long long ch = (N + ns - 1) / ns;
    ch = (ch + kTcTile - 1) / kTcTile * kTcTile;
    DecodePlan p;
    p.chunk = static_cast<int>(ch);
    p.nsplit = static_cast<int>((N + ch - 1) / ch);
    return p;
  }
  // CUDA-core path: the chunk's scores (chunk x gp floats) fit the score
  // buffer; at most 1024 keys.
  const int tile = kDecTile;
  int cmax = (kDecScoreBytes / 4 / gp) / kDecTile * kDecTile;
  if (cmax > 1024) cmax = 1024;
  // Enough CTAs to fill 4 per SM on 152 SMs where the keys allow chunks of at
  // least 256.
  long long want = (4 * 152 + units - 1) / units;
  const long long by_min = (N + 255) / 256;
  if (want > by_min) want = by_min;
  long long nsplit = (N + cmax - 1) / cmax;
  if (nsplit < want) nsplit = want;
  if (nsplit < 1) nsplit = 1;
  long long chunk = (N + nsplit - 1) / nsplit;
  chunk = (chunk + tile - 1) / tile * tile;
  DecodePlan p;
  p.chunk = static_cast<int>(chunk);
  p.nsplit = static_cast<int>((N + chunk - 1) / chunk);
  return p;
}

size_t decode_workspace_bytes(int B, int H, int Hkv, int N, int d) {
  const DecodePlan p = decode_plan(B, H, Hkv, N, d);
  return static_cast<size_t>(B) * H * p.nsplit * (d + 4) * sizeof(float);
}

fa_status launch_decode(const DecodeArgs& a, cudaStream_t s) {
  const DecodePlan p = decode_plan(a.B, a.H, a.Hkv, a.N, a.d);
  const int g = a.H / a.Hkv;
  if (use_tc(g, a.d)) return launch_decode_tc(a, p, s);
  // one query head per key/value head: the CUDA-core kernel
  return a.d == 64 ? launch_decode_impl<64, 1>(a, p, s) : launch_decode_impl<128, 1>(a, p, s);
}

uint32_t decode_take_error(cudaStream_t s) {
  uint32_t v = 0, zero = 0;
  cudaMemcpyFromSymbolAsync(&v, g_err_dec, sizeof(v), 0, cudaMemcpyDeviceToHost, s);
  cudaStreamSynchronize(s);
  cudaMemcpyToSymbolAsync(g_err_dec, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
  cudaStreamSynchronize(s);
  return v;
}

}  // namespace fa
