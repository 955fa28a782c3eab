// The C ABI declared in include/fa.h: argument checks, TMA tensor-map
// encoding, and the launch sequence of each entry point on the caller's stream.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa_common.cuh"
#include "fa_host.h"

namespace fa {

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn resolve_encode() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status check_shape(int B, int H, int N, int d) {
  if (B <= 0 || H <= 0 || N <= 0) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long bh = static_cast<long long>(B) * H;
  if (bh * N > (1LL << 31) / 1 || bh > (1LL << 30)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

fa_status check_scale(float scale) {
  return (std::isfinite(scale) && scale > 0.f) ? FA_OK : FA_ERR_INVALID_ARG;
}

fa_status check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_UNSUPPORTED;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  return (major == 10 && minor == 3) ? FA_OK : FA_ERR_UNSUPPORTED;
}

template <typename... P>
fa_status check_ptrs(P... ptrs) {
  const void* list[] = {static_cast<const void*>(ptrs)...};
  for (const void* p : list)
    if (p == nullptr) return FA_ERR_INVALID_ARG;
  for (const void* p : list)
    if (!aligned16(p)) return FA_ERR_ALIGNMENT;
  return FA_OK;
}

size_t round16(size_t x) { return (x + 15) & ~size_t(15); }

// ---------------------------------------------------------------- timeout hook

__device__ uint32_t g_err_probe;

__global__ void timeout_probe_kernel(long long limit_cycles) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  // Nothing ever arrives on `bar`: the wait below must run out and report.
  const long long t0 = clock64();
  while (!mbar_try_wait(&bar, 0)) {
    if (clock64() - t0 > limit_cycles) {
      atomicOr(&g_err_probe, FA_DEVERR_TIMEOUT);
      return;
    }
  }
}

}  // namespace

bool encode_rows_map(CUtensorMap* map, const void* base, int elem_bytes, int cols, int N, int BH, int box_cols,
                     int box_rows, int swizzle_bytes) {
  EncodeTiledFn enc = resolve_encode();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(N),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(cols) * elem_bytes,
                                 static_cast<cuuint64_t>(cols) * elem_bytes * static_cast<cuuint64_t>(N)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = elem_bytes == 4   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const CUtensorMapSwizzle swz = swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  return enc(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Special-function-unit rate: every thread runs 8 independent chains
// x <- 0.5 - 2^x (each step one ex2 and one FMA; x stays in [-1, 0.5]).  One
// CTA's cycle count is taken between two CTA barriers, so the rate is per SM
// with every CTA of the SM running.
__global__ void __launch_bounds__(512) ex2_rate_kernel(int iters, float* sink, long long* cycles) {
  float x[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) x[c] = -0.125f * static_cast<float>((threadIdx.x + c) & 7);
  __syncthreads();
  const long long t0 = clock64();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int c = 0; c < 8; ++c) x[c] = fmaf(-1.0f, ex2_approx(x[c]), 0.5f);
  }
  __syncthreads();
  const long long t1 = clock64();
  float acc = 0.f;
#pragma unroll
  for (int c = 0; c < 8; ++c) acc += x[c];
  sink[blockIdx.x * blockDim.x + threadIdx.x] = acc;
  if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

fa_status launch_ex2_rate(int blocks, int iters, float* sink, long long* cycles, cudaStream_t stream) {
  ex2_rate_kernel<<<blocks, 512, 0, stream>>>(iters, sink, cycles);
  return cudaPeekAtLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

// The polynomial exp2 of fa_common.cuh over an array (test hook): each thread
// takes two elements, the packed pair the kernels evaluate it on.
template <int DEG>
__global__ void __launch_bounds__(256) exp2_poly_kernel(const float* __restrict__ x, float* __restrict__ y,
                                                        long long n) {
  const long long i = 2 * (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const float x1 = i + 1 < n ? x[i + 1] : 0.0f;
  const float2 r = exp2_poly2<DEG>(make_float2(x[i], x1));
  y[i] = r.x;
  if (i + 1 < n) y[i + 1] = r.y;
}

fa_status launch_exp2_poly(const float* x, float* y, long long n, int degree, cudaStream_t stream) {
  const long long blocks = (n + 511) / 512;
  if (blocks > 0x7fffffffLL) return FA_ERR_INVALID_ARG;
  if (degree == 2)
    exp2_poly_kernel<2><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(x, y, n);
  else
    exp2_poly_kernel<3><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(x, y, n);
  return cudaPeekAtLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

// Scratch of the exp2-rate measurement: the sink (one float per thread) and
// one cycle count per CTA, for two CTAs of 512 threads per SM.
size_t ex2_rate_scratch_bytes(int sms) {
  const size_t blocks = 2 * static_cast<size_t>(sms);
  return round16(blocks * 512 * sizeof(float)) + blocks * sizeof(long long);
}

fa_status launch_timeout_probe(unsigned int limit_us, cudaStream_t stream) {
  int dev = 0, khz = 2000000;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev);
  const long long cycles = static_cast<long long>(limit_us) * (khz / 1000);
  timeout_probe_kernel<<<1, 32, 0, stream>>>(cycles);
  return cudaPeekAtLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

uint32_t probe_take_error(cudaStream_t s) {
  uint32_t v = 0, zero = 0;
  cudaMemcpyFromSymbolAsync(&v, g_err_probe, sizeof(v), 0, cudaMemcpyDeviceToHost, s);
  cudaStreamSynchronize(s);
  cudaMemcpyToSymbolAsync(g_err_probe, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s);
  cudaStreamSynchronize(s);
  return v;
}

}  // namespace fa

using namespace fa;

extern "C" {

namespace {

fa_status fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int N,
                     int d, int causal, int window, float scale, void* stream) {
  fa_status st;
  if ((st = check_ptrs(q, k, v, o, lse)) != FA_OK) return st;
  if ((st = check_shape(B, H, N, d)) != FA_OK) return st;
  if (Hkv <= 0 || H % Hkv != 0 || window < 0) return FA_ERR_INVALID_ARG;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if ((st = check_device()) != FA_OK) return st;
  FwdArgs a{q, k, v, o, lse, nullptr, nullptr, nullptr, B, H, N, d, causal, scale, Hkv, window};
  return launch_fwd_bf16(a, static_cast<cudaStream_t>(stream));
}

fa_status bwd_common(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                     void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                     int N, int d, int causal, int window, float scale, void* stream);

}  // namespace

fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv, int N,
                     int d, int causal, float scale, void* stream) {
  return fwd_common(q, k, v, o, lse, B, H, Hkv, N, d, causal, 0, scale, stream);
}

fa_status fa_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Hkv,
                        int N, int d, int window, float scale, void* stream) {
  if (window <= 0) return FA_ERR_INVALID_ARG;
  return fwd_common(q, k, v, o, lse, B, H, Hkv, N, d, 1, window >= N ? 0 : window, scale, stream);
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                 int causal, float scale, void* stream) {
  return fa_fwd_gqa(q, k, v, o, lse, B, H, H, N, d, causal, scale, stream);
}

size_t fa_bwd_workspace_size(int B, int H, int N, int d) {
  if (check_shape(B, H, N, d) != FA_OK) return 0;
  const size_t rows = static_cast<size_t>(B) * H * N;
  return round16(rows * sizeof(float)) + rows * d * sizeof(float);
}

namespace {

// Grouped-query backward with one CTA per query head (partial dK and dV added
// into fp32 accumulators) rather than per key/value head, whose CTAs walk every
// query head of their group one after the other: for groups of four query
// heads or more, or when the key/value heads give fewer than two waves of CTAs
// on 152 SMs.  Measured at B=2, H=32, N=8192, d=128, causal: groups of 2 lose
// 8 % split, of 4 gain 2 %, of 8 gain 12 %, of 32 (one key/value head) 2x.
bool bwd_split_heads(int B, int H, int Hkv, int N) {
  if (Hkv <= 0 || H % Hkv != 0 || Hkv == H) return false;
  const long long ctas = static_cast<long long>(B) * Hkv * ((N + 127) / 128);
  return H / Hkv >= 4 || ctas < 2 * 152;
}

size_t kv_acc_bytes(int B, int Hkv, int N, int d) {
  return round16(static_cast<size_t>(B) * Hkv * N * d * sizeof(float));
}

}  // namespace

size_t fa_bwd_gqa_workspace_size(int B, int H, int Hkv, int N, int d) {
  const size_t base = fa_bwd_workspace_size(B, H, N, d);
  if (base == 0 || Hkv <= 0 || H % Hkv != 0) return 0;
  return bwd_split_heads(B, H, Hkv, N) ? base + 2 * kv_acc_bytes(B, Hkv, N, d) : base;
}

fa_status fa_bwd_preprocess(const void* o, const void* dO, float* D, float* dq_acc, int B, int H, int N, int d,
                            void* stream) {
  fa_status st;
  if ((st = check_ptrs(o, dO, D, dq_acc)) != FA_OK) return st;
  if ((st = check_shape(B, H, N, d)) != FA_OK) return st;
  if ((st = check_device()) != FA_OK) return st;
  return launch_bwd_preprocess(o, dO, D, dq_acc, static_cast<long long>(B) * H * N, d,
                               static_cast<cudaStream_t>(stream));
}

fa_status fa_bwd_main(const void* q, const void* k, const void* v, const float* lse, const void* dO,
                      const float* D, float* dq_acc, void* dk, void* dv, int B, int H, int N, int d, int causal,
                      float scale, void* stream) {
  fa_status st;
  if ((st = check_ptrs(q, k, v, lse, dO, D, dq_acc, dk, dv)) != FA_OK) return st;
  if ((st = check_shape(B, H, N, d)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if ((st = check_device()) != FA_OK) return st;
  BwdArgs a{q, k, v, lse, dO, D, dq_acc, dk, dv, B, H, N, d, causal, scale, H};
  return launch_bwd_main(a, static_cast<cudaStream_t>(stream));
}

fa_status fa_bwd_dq_convert(const float* dq_acc, void* dq, int B, int H, int N, int d, float scale, void* stream) {
  fa_status st;
  if ((st = check_ptrs(dq_acc, dq)) != FA_OK) return st;
  if ((st = check_shape(B, H, N, d)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if ((st = check_device()) != FA_OK) return st;
  return launch_bwd_dq_convert(dq_acc, dq, static_cast<long long>(B) * H * N, d, scale,
                               static_cast<cudaStream_t>(stream));
}

namespace {

fa_status bwd_common(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                     void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                     int N, int d, int causal, int window, float scale, void* stream) {
  fa_status st;
  if ((st = check_ptrs(q, k, v, o, lse, dO, dq, dk, dv)) != FA_OK) return st;
  if ((st = check_shape(B, H, N, d)) != FA_OK) return st;
  if (Hkv <= 0 || H % Hkv != 0 || window < 0) return FA_ERR_INVALID_ARG;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  const size_t need = fa_bwd_workspace_size(B, H, N, d);
  if (workspace == nullptr || workspace_bytes < need) return FA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return FA_ERR_ALIGNMENT;
  if ((st = check_device()) != FA_OK) return st;
  const size_t rows = static_cast<size_t>(B) * H * N;
  float* Dvec = static_cast<float*>(workspace);
  float* dq_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + round16(rows * sizeof(float)));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // One CTA per query head when the workspace has room for the dK and dV
  // accumulators (fa_bwd_gqa_workspace_size) and the heads call for it.
  const size_t acc = kv_acc_bytes(B, Hkv, N, d);
  const bool split = window == 0 && bwd_split_heads(B, H, Hkv, N) && workspace_bytes >= need + 2 * acc;
  float* dk_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + need);
  float* dv_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + need + acc);
  if (split && cudaMemsetAsync(dk_acc, 0, 2 * acc, s) != cudaSuccess) return FA_ERR_LAUNCH;
  if ((st = launch_bwd_preprocess(o, dO, Dvec, dq_acc, static_cast<long long>(rows), d, s)) != FA_OK) return st;
  BwdArgs a{q, k, v, lse, dO, Dvec, dq_acc, split ? static_cast<void*>(dk_acc) : dk,
            split ? static_cast<void*>(dv_acc) : dv, B, H, N, d, causal, scale, Hkv, window, split};
  if ((st = launch_bwd_main(a, s)) != FA_OK) return st;
  if ((st = launch_bwd_dq_convert(dq_acc, dq, static_cast<long long>(rows), d, scale, s)) != FA_OK) return st;
  if (split) {
    const long long kv_rows = static_cast<long long>(B) * Hkv * N;
    if ((st = launch_bwd_dq_convert(dk_acc, dk, kv_rows, d, 1.0f, s)) != FA_OK) return st;
    if ((st = launch_bwd_dq_convert(dv_acc, dv, kv_rows, d, 1.0f, s)) != FA_OK) return st;
  }
  return FA_OK;
}

}  // namespace

fa_status fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                     void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                     int N, int d, int causal, float scale, void* stream) {
  return bwd_common(q, k, v, o, lse, dO, dq, dk, dv, workspace, workspace_bytes, B, H, Hkv, N, d, causal, 0, scale,
                    stream);
}

fa_status fa_bwd_window(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                        void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int Hkv,
                        int N, int d, int window, float scale, void* stream) {
  if (window <= 0) return FA_ERR_INVALID_ARG;
  return bwd_common(q, k, v, o, lse, dO, dq, dk, dv, workspace, workspace_bytes, B, H, Hkv, N, d, 1,
                    window >= N ? 0 : window, scale, stream);
}

fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                 void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int H, int N, int d,
                 int causal, float scale, void* stream) {
  return fa_bwd_gqa(q, k, v, o, lse, dO, dq, dk, dv, workspace, workspace_bytes, B, H, H, N, d, causal, scale,
                    stream);
}

fa_status fa_fwd_fp8(const void* q8, const void* k8, const void* v8, const float* descale_q,
                     const float* descale_k, const float* descale_v, void* o, float* lse, int B, int H, int N,
                     int d, int causal, float scale, void* stream) {
  fa_status st;
  if ((st = check_ptrs(q8, k8, v8, o, lse)) != FA_OK) return st;
  if (descale_q == nullptr || descale_k == nullptr || descale_v == nullptr) return FA_ERR_INVALID_ARG;
  if ((st = check_shape(B, H, N, d)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if ((st = check_device()) != FA_OK) return st;
  FwdArgs a{q8, k8, v8, o, lse, descale_q, descale_k, descale_v, B, H, N, d, causal, scale, H};
  return launch_fwd_fp8(a, static_cast<cudaStream_t>(stream));
}

fa_status fa_fwd_fp8_blocks(const void* q8, const void* k8, const void* v8, const float* descale_q,
                            const float* descale_k, const float* descale_v, void* o, float* lse, int B, int H,
                            int N, int d, int causal, float scale, void* stream) {
  fa_status st;
  if ((st = check_ptrs(q8, k8, v8, o, lse)) != FA_OK) return st;
  if (descale_q == nullptr || descale_k == nullptr || descale_v == nullptr) return FA_ERR_INVALID_ARG;
  if ((st = check_shape(B, H, N, d)) != FA_OK) return st;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if ((st = check_device()) != FA_OK) return st;
  FwdArgs a{q8, k8, v8, o, lse, descale_q, descale_k, descale_v, B, H, N, d, causal, scale, H};
  return launch_fwd_fp8_blocks(a, static_cast<cudaStream_t>(stream));
}

fa_status fa_fp8_quantize_blocks(const void* x, int x_dtype, int hadamard, int block_rows, void* codes,
                                 float* descale, int seqs, int N, int d, void* stream) {
  fa_status st;
  if ((st = check_ptrs(x, codes, descale)) != FA_OK) return st;
  if (seqs <= 0 || seqs > 65535 || N <= 0 || block_rows <= 0 || block_rows > 1024 || (x_dtype != 0 && x_dtype != 1) ||
      (hadamard != 0 && hadamard != 1) || static_cast<long long>(seqs) * N > (1LL << 31))
    return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if ((st = check_device()) != FA_OK) return st;
  return launch_fp8_quantize_blocks(x, x_dtype, hadamard, block_rows, codes, descale, seqs, N, d,
                                    static_cast<cudaStream_t>(stream));
}

size_t fa_decode_workspace_size(int B, int H, int Hkv, int N, int d) {
  if (B <= 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || N <= 0 || (d != 64 && d != 128)) return 0;
  return round16(decode_workspace_bytes(B, H, Hkv, N, d));
}

fa_status fa_decode(const void* q, const void* k, const void* v, void* o, float* lse, void* workspace,
                    size_t workspace_bytes, int B, int H, int Hkv, int N, int d, float scale, void* stream) {
  fa_status st;
  if ((st = check_ptrs(q, k, v, o, lse)) != FA_OK) return st;
  if (B <= 0 || H <= 0 || N <= 0 || Hkv <= 0 || H % Hkv != 0 || H / Hkv > 16 || B > 65535 ||
      static_cast<long long>(B) * Hkv > 65535)
    return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if ((st = check_scale(scale)) != FA_OK) return st;
  if (workspace == nullptr || workspace_bytes < fa_decode_workspace_size(B, H, Hkv, N, d))
    return FA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return FA_ERR_ALIGNMENT;
  if ((st = check_device()) != FA_OK) return st;
  DecodeArgs a{q, k, v, o, lse, static_cast<float*>(workspace), B, H, Hkv, N, d, scale};
  return launch_decode(a, static_cast<cudaStream_t>(stream));
}

fa_status fa_fp8_quantize(const void* x, int x_dtype, int hadamard, void* codes, float* descale, long long rows,
                          int d, void* stream) {
  fa_status st;
  if ((st = check_ptrs(x, codes, descale)) != FA_OK) return st;
  if (rows <= 0 || rows > (1LL << 31) || (x_dtype != 0 && x_dtype != 1) || (hadamard != 0 && hadamard != 1))
    return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if ((st = check_device()) != FA_OK) return st;
  return launch_fp8_quantize(x, x_dtype, hadamard, codes, descale, rows, d, static_cast<cudaStream_t>(stream));
}

const char* fa_status_string(fa_status s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: null pointer, non-positive size or bad scale";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: head dim or device not supported";
    case FA_ERR_ALIGNMENT: return "FA_ERR_ALIGNMENT: a pointer is not 16-byte aligned";
    case FA_ERR_LAUNCH: return "FA_ERR_LAUNCH: kernel launch or tensor-map encoding failed";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a kernel wait ran past its limit";
    case FA_ERR_WORKSPACE: return "FA_ERR_WORKSPACE: workspace missing or too small";
    case FA_ERR_KERNEL_CONFIG:
      return "FA_ERR_KERNEL_CONFIG: the compiled kernel's register count differs from its launch plan";
  }
  return "unknown fa_status";
}

fa_status fa_device_error(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_LAUNCH;
  uint32_t e = fwd_bf16_take_error(s) | bwd_take_error(s) | probe_take_error(s) | decode_take_error(s);
  if (cudaStreamSynchronize(s) != cudaSuccess) return FA_ERR_LAUNCH;
  if (e & FA_DEVERR_TIMEOUT) return FA_ERR_TIMEOUT;
  if (e != 0) return FA_ERR_LAUNCH;
  return FA_OK;
}

size_t fa_measure_ex2_rate_scratch_size(void) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return 0;
  return ex2_rate_scratch_bytes(sms);
}

fa_status fa_measure_ex2_rate(float* ex2_per_clock_per_sm, void* scratch, size_t scratch_bytes, void* stream) {
  fa_status st;
  if (ex2_per_clock_per_sm == nullptr || scratch == nullptr) return FA_ERR_INVALID_ARG;
  if (!aligned16(scratch)) return FA_ERR_ALIGNMENT;
  if ((st = check_device()) != FA_OK) return st;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0 || scratch_bytes < ex2_rate_scratch_bytes(sms)) return FA_ERR_WORKSPACE;
  const int blocks = 2 * sms, iters = 4096;  // two CTAs of 512 threads per SM
  float* sink = static_cast<float*>(scratch);
  long long* cycles = reinterpret_cast<long long*>(static_cast<char*>(scratch) +
                                                   round16(static_cast<size_t>(blocks) * 512 * sizeof(float)));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = launch_ex2_rate(blocks, iters, sink, cycles, s);  // warm-up
  if (st == FA_OK) st = launch_ex2_rate(blocks, iters, sink, cycles, s);
  long long* host = new long long[blocks];
  if (st == FA_OK && (cudaMemcpyAsync(host, cycles, sizeof(long long) * blocks, cudaMemcpyDeviceToHost, s) !=
                          cudaSuccess ||
                      cudaStreamSynchronize(s) != cudaSuccess))
    st = FA_ERR_LAUNCH;
  if (st == FA_OK) {
    long long worst = 1;
    for (int b = 0; b < blocks; ++b) worst = host[b] > worst ? host[b] : worst;
    // two CTAs per SM shared the SM for `worst` cycles
    *ex2_per_clock_per_sm = static_cast<float>(2.0 * 512.0 * 8.0 * iters / static_cast<double>(worst));
  }
  delete[] host;
  return st;
}

fa_status fa_debug_exp2_poly(const float* x, float* y, long long n, int degree, void* stream) {
  fa_status st;
  if ((st = check_ptrs(x, y)) != FA_OK) return st;
  if (n <= 0 || (degree != 2 && degree != 3)) return FA_ERR_INVALID_ARG;
  if ((st = check_device()) != FA_OK) return st;
  return launch_exp2_poly(x, y, n, degree, static_cast<cudaStream_t>(stream));
}

fa_status fa_debug_wait_timeout(unsigned int limit_us, void* stream) {
  if (limit_us < 1 || limit_us > 1000000) return FA_ERR_INVALID_ARG;
  fa_status st;
  if ((st = check_device()) != FA_OK) return st;
  return launch_timeout_probe(limit_us, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
