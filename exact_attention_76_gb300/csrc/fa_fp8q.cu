// Per-tensor e4m3 storage for the FP8 forward, with optional incoherent
// processing ("FLASH-ATTN", FlashAttention-3 > Low-precision with FP8: one
// scale per tensor; Q and K multiplied by an orthogonal matrix M before
// quantisation, which leaves (QM)(KM)^T = QK^T and spreads outliers;
// "FlashAttention 三代演进", 技术 4: M is a Hadamard transform).
//
//   y      = x H / sqrt(d)     (if rotating; H the Sylvester Hadamard matrix)
//   delta  = max |y| / 448     (one fp32 per tensor, 448 = largest e4m3)
//   code   = e4m3_rne(y / delta)
//
// Two layouts of the work:
//  * lane-split (no rotation, and rotated blocks of more than 128 rows): one
//    warp per row of d values (d / 32 per lane, one vector load, several rows
//    in flight); the rotation there is a fast Walsh-Hadamard transform whose
//    butterflies (a, b) -> (a + b, a - b) run over the index bits, first those
//    inside a lane's registers, then the lane bits through warp shuffles;
//  * row per lane (every other rotated input): a warp stages 32 rows in
//    shared memory and each lane transforms a whole row in registers, the
//    same butterflies in the same order.
// Per tensor: three launches -- max |y| (atomic max on the float's bit
// pattern, valid for non-negative floats), the codes, and delta, the last two
// launched while the one before finishes.  Per block (block quantisation of
// the same section: blocks of B_r x d or B_c x d rows, one scale each): one
// launch, one CTA per block; fp32 blocks of up to 128 rows are held in
// registers, other unrotated blocks read twice (the second time from L1).
// Every code is y * 448 / max|y| rounded once to fp32 (code_scale below).
#include <cuda_bf16.h>

#include "fa_common.cuh"
#include "fa_host.h"

namespace fa {

namespace {

// This lane's d / 32 values of a row, in one vector load (x is 16-byte
// aligned, so every lane's part is aligned to its size).
template <int D, typename T>
__device__ __forceinline__ void load_row(const T* __restrict__ x, long long row, float (&v)[D / 32]) {
  constexpr int E = D / 32;
  const T* src = x + row * D + static_cast<int>(lane_id()) * E;
  if constexpr (sizeof(T) == 4) {
    if constexpr (E == 4) {
      const float4 t = __ldg(reinterpret_cast<const float4*>(src));
      v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    } else {
      const float2 t = __ldg(reinterpret_cast<const float2*>(src));
      v[0] = t.x; v[1] = t.y;
    }
  } else {
    if constexpr (E == 4) {
      const uint2 t = __ldg(reinterpret_cast<const uint2*>(src));
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&t.x));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&t.y));
      v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
    } else {
      const uint32_t t = __ldg(reinterpret_cast<const unsigned int*>(src));
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&t));
      v[0] = a.x; v[1] = a.y;
    }
  }
}

// y = x H / sqrt(d) of the row whose lane values are v.
template <int D>
__device__ __forceinline__ void rotate_row(float (&v)[D / 32]) {
  constexpr int E = D / 32;
  const int lane = static_cast<int>(lane_id());
  // index bits inside the lane: e = lane * E + j
#pragma unroll
  for (int h = 1; h < E; h <<= 1) {
#pragma unroll
    for (int j = 0; j < E; ++j) {
      if ((j & h) == 0) {
        const float a = v[j], b = v[j + h];
        v[j] = a + b;
        v[j + h] = a - b;
      }
    }
  }
  // index bits across lanes: partner element is e ^ (m * E), i.e. lane ^ m
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool high = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < E; ++j) {
      const float p = __shfl_xor_sync(0xffffffffu, v[j], m);
      v[j] = high ? (p - v[j]) : (v[j] + p);
    }
  }
  const float norm = rsqrtf(static_cast<float>(D));
#pragma unroll
  for (int j = 0; j < E; ++j) v[j] *= norm;
}

// y / delta as a product with a two-word reciprocal: inv_hi + inv_lo carries
// 448 / max|y| to about 2^-48 relative (inv_hi = RN(448 / A); the residual
// 448 - inv_hi A of a correctly rounded quotient is exact in one fma, and
// inv_lo is that residual over A), and code = e4m3(fma(y, inv_hi, y inv_lo))
// rounds y 448 / max|y| once.  A quotient that falls exactly on an e4m3
// midpoint -- common with bf16 input, whose short significands make ratios
// such as 21 = (25.5 / 448)^-1 x 1.1953125 exact -- stays exact and rounds to
// even, as in the float64 definition; the single-word reciprocal or a quotient
// by the rounded delta misses such a tie whenever their one rounding error
// exceeds half an ulp of the quotient.  Both words are computed once per kernel
// or block, so each code costs three operations instead of a division.
// pre = 2^100 scales a maximum below 2^-100 up (exactly: |y| <= max|y|) so
// that the reciprocal stays finite; an all-zero tensor or block has delta = 1
// (pre = inv_hi = 1, inv_lo = 0), and an infinite maximum gives inv = 0.
struct CodeScale {
  float pre, hi, lo;
};

__device__ __forceinline__ CodeScale code_scale(float amax) {
  if (!(amax > 0.f)) return {1.f, 1.f, 0.f};
  const float pre = amax < 0x1p-100f ? 0x1p100f : 1.f;
  const float a = amax * pre;
  const float hi = __fdiv_rn(448.0f, a);
  const float lo = a < INFINITY ? __fdiv_rn(__fmaf_rn(-hi, a, 448.0f), a) : 0.f;
  return {pre, hi, lo};
}

__device__ __forceinline__ float code_value(float y, CodeScale c) {
  const float s = y * c.pre;
  return __fmaf_rn(s, c.hi, s * c.lo);
}

// The per-tensor codes kernels are launched while the max|y| kernel before
// them finishes (programmatic dependent launch).  Their input x is only read
// (by both kernels), so a CTA loads its first rows first and waits for the
// maximum only when it needs the scale; the maximum itself is read after the
// wait with a plain (not read-only-cached) load.
__device__ __forceinline__ CodeScale scale_after_max_kernel(const unsigned int* amax_bits) {
  pdl_wait_prior();
  return code_scale(__uint_as_float(*reinterpret_cast<const volatile unsigned int*>(amax_bits)));
}

// This lane's 4 e4m3 codes (or 2 at d = 64) of y / delta, stored at dst.
template <int D>
__device__ __forceinline__ void store_codes(uint8_t* dst, const float (&v)[D / 32], CodeScale c) {
  if constexpr (D / 32 == 4) {
    *reinterpret_cast<uint32_t*>(dst) = pack_e4m3x4(code_value(v[0], c), code_value(v[1], c),
                                                    code_value(v[2], c), code_value(v[3], c));
  } else {
    const uint32_t w = pack_e4m3x4(code_value(v[0], c), code_value(v[1], c), 0.f, 0.f);
    *reinterpret_cast<uint16_t*>(dst) = static_cast<uint16_t>(w & 0xffffu);
  }
}

constexpr int kQRowsInFlight = 4;  // rows a warp loads before working on them
// The per-tensor kernels keep twice as many fp32 rows in flight (measured on
// 1 x 16 x 16384 x 128, L2 flushed: fp32 59.9 -> 56.9 us a call; bf16 ran
// 41.9 -> 45.7 with eight and keeps four).
template <typename T>
constexpr int kTensorRowsInFlight = sizeof(T) == 4 ? 2 * kQRowsInFlight : kQRowsInFlight;

template <int D, typename T>
__global__ void __launch_bounds__(256) fp8q_amax_kernel(const T* __restrict__ x, long long rows, int rotate,
                                                        unsigned int* __restrict__ amax_bits) {
  constexpr int E = D / 32, U = kTensorRowsInFlight<T>;
  pdl_launch_dependents();
  const long long warps = static_cast<long long>(gridDim.x) * 8;
  float m = 0.f;
  for (long long row0 = static_cast<long long>(blockIdx.x) * 8 + warp_id(); row0 < rows; row0 += U * warps) {
    float v[U][E];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long row = row0 + u * warps;
      if (row < rows) {
        load_row<D>(x, row, v[u]);
      } else {
#pragma unroll
        for (int j = 0; j < E; ++j) v[u][j] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (rotate) rotate_row<D>(v[u]);
#pragma unroll
      for (int j = 0; j < E; ++j) m = fmaxf(m, fabsf(v[u][j]));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  // the CTA's maximum first: one atomic per CTA on the shared word
  __shared__ float s_part[8];
  if (lane_id() == 0) s_part[warp_id()] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 1; i < 8; ++i) m = fmaxf(m, s_part[i]);
    atomicMax(amax_bits, __float_as_uint(m));
  }
}

template <int D, typename T>
__global__ void __launch_bounds__(256) fp8q_codes_kernel(const T* __restrict__ x, long long rows, int rotate,
                                                         const unsigned int* amax_bits,
                                                         uint8_t* __restrict__ codes) {
  constexpr int E = D / 32, U = kTensorRowsInFlight<T>;
  pdl_launch_dependents();
  CodeScale cs{};
  bool have_scale = false;
  const long long warps = static_cast<long long>(gridDim.x) * 8;
  for (long long row0 = static_cast<long long>(blockIdx.x) * 8 + warp_id(); row0 < rows; row0 += U * warps) {
    float v[U][E];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (row0 + u * warps < rows) load_row<D>(x, row0 + u * warps, v[u]);
    if (!have_scale) {
      cs = scale_after_max_kernel(amax_bits);
      have_scale = true;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const long long row = row0 + u * warps;
      if (row < rows) {
        if (rotate) rotate_row<D>(v[u]);
        store_codes<D>(codes + row * D + lane_id() * E, v[u], cs);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// The rotated quantisers with one row per lane: a warp stages 32 rows in
// shared memory by asynchronous 16-byte copies, all in flight at once (rows
// padded by 16 bytes: a lane's 16-byte loads of its own row are then free of
// bank conflicts), and each lane transforms its row in registers -- the
// butterflies of rotate_row in the same order (index bit 0 first), so the
// results are the same to the bit, without the warp shuffles of the
// lane-split form.
template <int D, typename T>
constexpr int kRotRowElems = D + 16 / static_cast<int>(sizeof(T));
template <int D, typename T>
constexpr int kRotWarpBytes = 32 * kRotRowElems<D, T> * static_cast<int>(sizeof(T));

// 16 bytes global -> shared, asynchronously; zero-filled when !valid (the
// source address is then not read).
__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(smem_dst)), "l"(gsrc),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Starts the copies of rows [row0, row0 + 32) (zeros past row_end) into the
// warp's staging buffer, as one committed group.
template <int D, typename T>
__device__ __forceinline__ void stage_rows(const T* __restrict__ x, long long row0, long long row_end,
                                           uint8_t* __restrict__ wbuf) {
  constexpr int VEC = 16 / static_cast<int>(sizeof(T));  // elements per 16-byte copy
  constexpr int STRIDE = kRotRowElems<D, T>;
  constexpr int CHUNKS = 32 * D / VEC;
  const int lane = static_cast<int>(lane_id());
  const long long avail = row_end - row0 >= 32 ? 32ll * D : (row_end > row0 ? (row_end - row0) * D : 0ll);
  const T* src = x + (row_end > row0 ? row0 : 0) * D;
  T* tb = reinterpret_cast<T*>(wbuf);
#pragma unroll
  for (int c = lane; c < CHUNKS; c += 32) {
    const int e = c * VEC;
    const bool valid = e < avail;
    cp_async16(tb + (e / D) * STRIDE + (e % D), valid ? src + e : src, valid);
  }
  cp_async_commit();
}

// Waits for the staged rows and moves this lane's row into v; the buffer is
// free for the next stage_rows when this returns.
template <int D, typename T>
__device__ __forceinline__ void take_row(const uint8_t* __restrict__ wbuf, float (&v)[D]) {
  constexpr int VEC = 16 / static_cast<int>(sizeof(T));
  constexpr int STRIDE = kRotRowElems<D, T>;
  cp_async_wait_all();
  __syncwarp();
  const T* mine = reinterpret_cast<const T*>(wbuf) + static_cast<int>(lane_id()) * STRIDE;
#pragma unroll
  for (int k = 0; k < D; k += VEC) {
    const uint4 t = *reinterpret_cast<const uint4*>(mine + k);
    if constexpr (sizeof(T) == 4) {
      v[k] = __uint_as_float(t.x); v[k + 1] = __uint_as_float(t.y);
      v[k + 2] = __uint_as_float(t.z); v[k + 3] = __uint_as_float(t.w);
    } else {
      const uint32_t w4[4] = {t.x, t.y, t.z, t.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[i]));
        v[k + 2 * i] = p.x;
        v[k + 2 * i + 1] = p.y;
      }
    }
  }
  __syncwarp();
}

template <int D, typename T>
__device__ __forceinline__ void rows_to_lanes(const T* __restrict__ x, long long row0, long long row_end,
                                              uint8_t* __restrict__ wbuf, float (&v)[D]) {
  stage_rows<D, T>(x, row0, row_end, wbuf);
  take_row<D, T>(wbuf, v);
}

// y = x H / sqrt(d) of a whole row held by one lane.
template <int D>
__device__ __forceinline__ void rotate_own_row(float (&v)[D]) {
#pragma unroll
  for (int h = 1; h < D; h <<= 1) {
#pragma unroll
    for (int k = 0; k < D; ++k) {
      if ((k & h) == 0) {
        const float a = v[k], b = v[k + h];
        v[k] = a + b;
        v[k + h] = a - b;
      }
    }
  }
  const float norm = rsqrtf(static_cast<float>(D));
#pragma unroll
  for (int k = 0; k < D; ++k) v[k] *= norm;
}

// A lane's row of codes (d bytes) from y / delta.
template <int D>
__device__ __forceinline__ void store_own_codes(uint8_t* __restrict__ dst, const float (&v)[D], CodeScale c) {
#pragma unroll
  for (int k = 0; k < D; k += 16) {
    uint4 w;
    w.x = pack_e4m3x4(code_value(v[k], c), code_value(v[k + 1], c), code_value(v[k + 2], c),
                      code_value(v[k + 3], c));
    w.y = pack_e4m3x4(code_value(v[k + 4], c), code_value(v[k + 5], c), code_value(v[k + 6], c),
                      code_value(v[k + 7], c));
    w.z = pack_e4m3x4(code_value(v[k + 8], c), code_value(v[k + 9], c), code_value(v[k + 10], c),
                      code_value(v[k + 11], c));
    w.w = pack_e4m3x4(code_value(v[k + 12], c), code_value(v[k + 13], c), code_value(v[k + 14], c),
                      code_value(v[k + 15], c));
    *reinterpret_cast<uint4*>(dst + k) = w;
  }
}

constexpr int kRotWarps = 8;

template <int D, typename T>
__global__ void __launch_bounds__(kRotWarps * 32, 1) fp8q_amax_rot_kernel(const T* __restrict__ x, long long rows,
                                                                         unsigned int* __restrict__ amax_bits) {
  extern __shared__ float4 rot_smem[];
  pdl_launch_dependents();
  uint8_t* buf = reinterpret_cast<uint8_t*>(rot_smem) + warp_id() * kRotWarpBytes<D, T>;
  const long long step = static_cast<long long>(gridDim.x) * kRotWarps * 32;
  float m = 0.f;
  long long row0 = (static_cast<long long>(blockIdx.x) * kRotWarps + warp_id()) * 32;
  if (row0 < rows) stage_rows<D>(x, row0, rows, buf);
  for (; row0 < rows; row0 += step) {
    float v[D];
    take_row<D, T>(buf, v);
    if (row0 + step < rows) stage_rows<D>(x, row0 + step, rows, buf);  // in flight during the butterflies
    rotate_own_row<D>(v);
#pragma unroll
    for (int k = 0; k < D; ++k) m = fmaxf(m, fabsf(v[k]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  __shared__ float s_part[kRotWarps];
  if (lane_id() == 0) s_part[warp_id()] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int i = 1; i < kRotWarps; ++i) m = fmaxf(m, s_part[i]);
    atomicMax(amax_bits, __float_as_uint(m));
  }
}

template <int D, typename T>
__global__ void __launch_bounds__(kRotWarps * 32, 1) fp8q_codes_rot_kernel(const T* __restrict__ x, long long rows,
                                                                          const unsigned int* amax_bits,
                                                                          uint8_t* __restrict__ codes) {
  extern __shared__ float4 rot_smem[];
  pdl_launch_dependents();
  uint8_t* buf = reinterpret_cast<uint8_t*>(rot_smem) + warp_id() * kRotWarpBytes<D, T>;
  CodeScale cs{};
  bool have_scale = false;
  const long long step = static_cast<long long>(gridDim.x) * kRotWarps * 32;
  long long row0 = (static_cast<long long>(blockIdx.x) * kRotWarps + warp_id()) * 32;
  if (row0 < rows) stage_rows<D>(x, row0, rows, buf);
  for (; row0 < rows; row0 += step) {
    float v[D];
    take_row<D, T>(buf, v);
    if (row0 + step < rows) stage_rows<D>(x, row0 + step, rows, buf);
    rotate_own_row<D>(v);
    if (!have_scale) {
      cs = scale_after_max_kernel(amax_bits);
      have_scale = true;
    }
    const long long row = row0 + lane_id();
    if (row < rows) store_own_codes<D>(codes + row * D, v, cs);
  }
}

// Block storage with the rotation, blocks of at most 128 rows: one CTA per
// block with a warp per 32 of its rows (so 64-row blocks run two warps, not
// four of which two would rotate zeros), each lane one row, the block read
// once.
template <int D, typename T>
__global__ void __launch_bounds__(128) fp8qb_rot_kernel(const T* __restrict__ x, int N, int block_rows,
                                                        uint8_t* __restrict__ codes, float* __restrict__ descale) {
  extern __shared__ float4 rot_smem[];
  __shared__ float s_part[4];
  const int w = static_cast<int>(warp_id());
  uint8_t* buf = reinterpret_cast<uint8_t*>(rot_smem) + w * kRotWarpBytes<D, T>;
  const int blk = static_cast<int>(blockIdx.x);
  const long long seq = blockIdx.y;
  const long long base = seq * N;
  const int r0 = blk * block_rows;
  const int r1 = min(N, r0 + block_rows);
  const long long row0 = r0 + 32 * w;
  float v[D];
  rows_to_lanes<D>(x + base * D, row0, r1, buf, v);
  rotate_own_row<D>(v);
  float m = 0.f;
#pragma unroll
  for (int k = 0; k < D; ++k) m = fmaxf(m, fabsf(v[k]));  // rows past the block are zero
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane_id() == 0) s_part[w] = m;
  __syncthreads();
  float amax = s_part[0];
  for (int i = 1; i < static_cast<int>(blockDim.x >> 5); ++i) amax = fmaxf(amax, s_part[i]);
  if (threadIdx.x == 0) descale[seq * gridDim.x + blk] = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  const long long row = row0 + lane_id();
  if (row < r1) store_own_codes<D>(codes + (base + row) * D, v, code_scale(amax));
}

__global__ void fp8q_delta_kernel(float* __restrict__ descale) {
  pdl_wait_prior();
  const float amax = __uint_as_float(*reinterpret_cast<const unsigned int*>(descale));
  *descale = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
}

template <int D, typename T>
fa_status launch_impl(const void* x, int rotate, void* codes, float* descale, long long rows, cudaStream_t s) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long long blocks = (rows + 7) / 8;
  if (blocks > static_cast<long long>(sms) * 16) blocks = static_cast<long long>(sms) * 16;
  if (blocks < 1) blocks = 1;
  if (cudaMemsetAsync(descale, 0, sizeof(float), s) != cudaSuccess) return FA_ERR_LAUNCH;
  unsigned int* amax_bits = reinterpret_cast<unsigned int*>(descale);  // holds max |y| until the last step
  if (rotate) {
    // one row per lane: 32 rows a warp, one CTA of eight warps per SM
    // (measured on a 1 x 16 x 16384 x 128 input against the lane-split form:
    // with a division per code bf16 ran 1.39 TB/s against 1.28; with the
    // two-word reciprocal fp32 runs 2.29 against 2.21)
    const int smem = kRotWarps * kRotWarpBytes<D, T>;
    if (cudaFuncSetAttribute(fp8q_amax_rot_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess ||
        cudaFuncSetAttribute(fp8q_codes_rot_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
            cudaSuccess)
      return FA_ERR_LAUNCH;
    long long rblocks = (rows + kRotWarps * 32 - 1) / (kRotWarps * 32);
    if (rblocks > sms) rblocks = sms;
    fp8q_amax_rot_kernel<D, T><<<static_cast<unsigned>(rblocks), kRotWarps * 32, smem, s>>>(
        static_cast<const T*>(x), rows, amax_bits);
    if (launch_pdl(fp8q_codes_rot_kernel<D, T>, dim3(static_cast<unsigned>(rblocks)), dim3(kRotWarps * 32), smem,
                   s, static_cast<const T*>(x), rows, static_cast<const unsigned int*>(amax_bits),
                   static_cast<uint8_t*>(codes)) != cudaSuccess ||
        launch_pdl(fp8q_delta_kernel, dim3(1), dim3(1), 0, s, descale) != cudaSuccess)
      return FA_ERR_LAUNCH;
    return cudaPeekAtLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
  }
  fp8q_amax_kernel<D, T><<<static_cast<unsigned>(blocks), 256, 0, s>>>(static_cast<const T*>(x), rows, rotate,
                                                                        amax_bits);
  if (launch_pdl(fp8q_codes_kernel<D, T>, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                 static_cast<const T*>(x), rows, rotate, static_cast<const unsigned int*>(amax_bits),
                 static_cast<uint8_t*>(codes)) != cudaSuccess ||
      launch_pdl(fp8q_delta_kernel, dim3(1), dim3(1), 0, s, descale) != cudaSuccess)
    return FA_ERR_LAUNCH;
  return cudaPeekAtLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

// Block storage: one CTA per (block of block_rows rows, sequence).  With fp32
// input, up to 128 rows a block are held in registers (warp w takes rows w,
// w + 8, ..., all loaded before any is worked on) and read once; otherwise
// (bf16, and longer blocks) the block is read twice, for max |y| and for the
// codes, the second time mostly from L1, each warp with four rows in flight
// (measured on 1 x 16 x 16384 x 128, L2 flushed: bf16 128-row blocks 39.1 ->
// 32.8 us against one row in flight, 256-row fp32 blocks 62.4 -> 48.4 us; bf16
// held in registers ran 37.5).  Rotated blocks of up to 128 rows take the
// row-per-lane kernel above.
constexpr int kQbRowsPerWarp = 16;

// (The held form at three CTAs per SM: measured faster than at the two its
// unbounded register count allowed.)
template <int D, typename T, bool HELD>
__global__ void __launch_bounds__(256, HELD ? 3 : 1) fp8qb_kernel(const T* __restrict__ x, int N, int block_rows, int rotate,
                                                    uint8_t* __restrict__ codes, float* __restrict__ descale) {
  constexpr int E = D / 32, R = HELD ? kQbRowsPerWarp : 1;
  __shared__ float s_part[8];
  const int blk = static_cast<int>(blockIdx.x);
  const long long seq = blockIdx.y;
  const int r0 = blk * block_rows;
  const int r1 = min(N, r0 + block_rows);
  const long long base = seq * N;
  const int w = static_cast<int>(warp_id());
  float v[R][E];
  float m = 0.f;
  if constexpr (HELD) {
#pragma unroll
    for (int u = 0; u < R; ++u)
      if (r0 + w + 8 * u < r1) load_row<D>(x, base + r0 + w + 8 * u, v[u]);
#pragma unroll
    for (int u = 0; u < R; ++u) {
      if (r0 + w + 8 * u < r1) {
        if (rotate) rotate_row<D>(v[u]);
#pragma unroll
        for (int j = 0; j < E; ++j) m = fmaxf(m, fabsf(v[u][j]));
      }
    }
  } else {
    for (int row = r0 + w; row < r1; row += 8 * kQRowsInFlight) {
      float t[kQRowsInFlight][E];
#pragma unroll
      for (int u = 0; u < kQRowsInFlight; ++u) {
        if (row + 8 * u < r1) {
          load_row<D>(x, base + row + 8 * u, t[u]);
        } else {
#pragma unroll
          for (int j = 0; j < E; ++j) t[u][j] = 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < kQRowsInFlight; ++u) {
        if (rotate) rotate_row<D>(t[u]);
#pragma unroll
        for (int j = 0; j < E; ++j) m = fmaxf(m, fabsf(t[u][j]));
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane_id() == 0) s_part[w] = m;
  __syncthreads();
  float amax = s_part[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, s_part[i]);
  if (threadIdx.x == 0) descale[seq * gridDim.x + blk] = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  const CodeScale cs = code_scale(amax);
  if constexpr (HELD) {
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const int row = r0 + w + 8 * u;
      if (row < r1) store_codes<D>(codes + (base + row) * D + lane_id() * E, v[u], cs);
    }
  } else {
    for (int row = r0 + w; row < r1; row += 8 * kQRowsInFlight) {
      float t[kQRowsInFlight][E];
#pragma unroll
      for (int u = 0; u < kQRowsInFlight; ++u)
        if (row + 8 * u < r1) load_row<D>(x, base + row + 8 * u, t[u]);
#pragma unroll
      for (int u = 0; u < kQRowsInFlight; ++u) {
        if (row + 8 * u < r1) {
          if (rotate) rotate_row<D>(t[u]);
          store_codes<D>(codes + (base + row + 8 * u) * D + lane_id() * E, t[u], cs);
        }
      }
    }
  }
}

template <int D, typename T>
fa_status launch_blocks_impl(const void* x, int rotate, int block_rows, void* codes, float* descale, int seqs, int N,
                             cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((N + block_rows - 1) / block_rows), static_cast<unsigned>(seqs));
  if (rotate && block_rows <= 128) {  // one row per lane (measured: fp32 3.21 -> 3.31 TB/s, bf16 1.86 -> 2.40)
    const int smem = 4 * kRotWarpBytes<D, T>;
    if (cudaFuncSetAttribute(fp8qb_rot_kernel<D, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return FA_ERR_LAUNCH;
    const int warps = (block_rows + 31) / 32;
    fp8qb_rot_kernel<D, T><<<grid, 32 * warps, warps * kRotWarpBytes<D, T>, s>>>(
        static_cast<const T*>(x), N, block_rows, static_cast<uint8_t*>(codes), descale);
  } else {
    bool held = false;
    if constexpr (sizeof(T) == 4) {
      held = block_rows <= 8 * kQbRowsPerWarp;
      if (held)
        fp8qb_kernel<D, T, true><<<grid, 256, 0, s>>>(static_cast<const T*>(x), N, block_rows, rotate,
                                                      static_cast<uint8_t*>(codes), descale);
    }
    if (!held)
      fp8qb_kernel<D, T, false><<<grid, 256, 0, s>>>(static_cast<const T*>(x), N, block_rows, rotate,
                                                     static_cast<uint8_t*>(codes), descale);
  }
  return cudaPeekAtLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

}  // namespace

fa_status launch_fp8_quantize_blocks(const void* x, int x_dtype, int rotate, int block_rows, void* codes,
                                     float* descale, int seqs, int N, int d, cudaStream_t s) {
  if (d == 64)
    return x_dtype == 1 ? launch_blocks_impl<64, __nv_bfloat16>(x, rotate, block_rows, codes, descale, seqs, N, s)
                        : launch_blocks_impl<64, float>(x, rotate, block_rows, codes, descale, seqs, N, s);
  return x_dtype == 1 ? launch_blocks_impl<128, __nv_bfloat16>(x, rotate, block_rows, codes, descale, seqs, N, s)
                      : launch_blocks_impl<128, float>(x, rotate, block_rows, codes, descale, seqs, N, s);
}

fa_status launch_fp8_quantize(const void* x, int x_dtype, int rotate, void* codes, float* descale, long long rows,
                              int d, cudaStream_t s) {
  if (d == 64)
    return x_dtype == 1 ? launch_impl<64, __nv_bfloat16>(x, rotate, codes, descale, rows, s)
                        : launch_impl<64, float>(x, rotate, codes, descale, rows, s);
  return x_dtype == 1 ? launch_impl<128, __nv_bfloat16>(x, rotate, codes, descale, rows, s)
                      : launch_impl<128, float>(x, rotate, codes, descale, rows, s);
}

}  // namespace fa
