// Host-side helpers shared by the launchers: TMA tensor-map encoding through
// the driver entry point, argument structs and the launcher declarations.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/fa.h"

namespace fa {

// Encodes a 3-D tiled map over a [BH, N, cols] row-major tensor of
// `elem_bytes`-byte elements with a box of (box_cols x box_rows x 1) and the
// 128-byte swizzle (64-byte when swizzle_bytes is 64; the box row must then be
// 64 bytes).  Rows past N read as zeros.  Returns false on failure.
bool encode_rows_map(CUtensorMap* map, const void* base, int elem_bytes, int cols, int N, int BH, int box_cols,
                     int box_rows, int swizzle_bytes = 128);

// Launches `kern` on `stream` with programmatic stream serialization: the
// kernel may begin launching while the previous kernel of the stream is still
// finishing (its set-up overlaps that kernel's last CTAs) and waits for it
// with griddepcontrol.wait before touching memory.  Used for the forward and
// backward main kernels, whose CTAs need a whole SM and so never sit beside
// the previous kernel's CTAs: measured, the fwd+bwd step of the GPT-2-small
// layer (B=4, H=12, N=1024, d=64) went from 65.7 to 57.7 us causal, the long
// causal one (B=2, H=16, N=8192, d=128) stayed the same.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  const float* descale_q;  // FP8 only (device pointers): one value, or one per block
  const float* descale_k;
  const float* descale_v;
  int B, H, N, d;
  int causal;
  float scale;
  int Hkv;  // key/value heads; H % Hkv == 0 (H for plain multi-head attention)
  int window = 0;  // causal sliding window of this many keys (0: none)
};

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const float* lse;
  const void* dO;
  const float* D;
  float* dq_acc;
  void* dk;
  void* dv;
  int B, H, N, d;
  int causal;
  float scale;
  int Hkv;  // key/value heads of k, v, dk, dv; H % Hkv == 0
  int window = 0;  // causal sliding window of this many keys (0: none)
  // dk and dv are fp32 accumulators (zeroed) into which one CTA per query
  // head adds its part (grouped-query heads; not with a window)
  bool split_heads = false;
};

fa_status launch_fwd_bf16(const FwdArgs& a, cudaStream_t stream);
fa_status launch_fwd_fp8(const FwdArgs& a, cudaStream_t stream);
struct DecodeArgs {
  const void* q;  // [B, H, d] bf16
  const void* k;  // [B, Hkv, N, d] bf16
  const void* v;
  void* o;        // [B, H, d] bf16
  float* lse;     // [B, H]
  float* part;    // workspace: per (row, chunk) d + 4 floats
  int B, H, Hkv, N, d;
  float scale;
};

struct DecodePlan {
  int chunk;   // keys per CTA (multiple of 64)
  int nsplit;  // chunks per key/value head
};

DecodePlan decode_plan(int B, int H, int Hkv, int N, int d);
size_t decode_workspace_bytes(int B, int H, int Hkv, int N, int d);
fa_status launch_decode(const DecodeArgs& a, cudaStream_t stream);
uint32_t decode_take_error(cudaStream_t s);

fa_status launch_bwd_preprocess(const void* o, const void* dO, float* D, float* dq_acc, long long rows, int d,
                                cudaStream_t stream);
fa_status launch_bwd_main(const BwdArgs& a, cudaStream_t stream);
fa_status launch_bwd_dq_convert(const float* dq_acc, void* dq, long long rows, int d, float scale,
                                cudaStream_t stream);
fa_status launch_timeout_probe(unsigned int limit_us, cudaStream_t stream);
fa_status launch_fp8_quantize(const void* x, int x_dtype, int rotate, void* codes, float* descale, long long rows,
                              int d, cudaStream_t stream);
fa_status launch_fp8_quantize_blocks(const void* x, int x_dtype, int rotate, int block_rows, void* codes,
                                     float* descale, int seqs, int N, int d, cudaStream_t stream);
fa_status launch_fwd_fp8_blocks(const FwdArgs& a, cudaStream_t stream);

// Reads and clears each translation unit's device error word (stream-ordered
// copy followed by a stream synchronisation done by the caller).
uint32_t fwd_bf16_take_error(cudaStream_t s);
uint32_t fwd_fp8_take_error(cudaStream_t s);
uint32_t bwd_take_error(cudaStream_t s);
uint32_t probe_take_error(cudaStream_t s);

}  // namespace fa
