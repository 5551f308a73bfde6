// common.cuh -- definitions shared by the CUDA translation units of
// libattnprefill.so: problem constants, the launch-parameter block, the
// device error word protocol and the host-side launcher declarations.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/attn_prefill.h"

namespace attn {

constexpr int kHQ = ATTN_HQ;            // query heads
constexpr int kHKV = ATTN_HKV;          // KV heads
constexpr int kGroup = kHQ / kHKV;      // query heads per KV head (4)
constexpr int kD = ATTN_D;              // head dimension
constexpr float kScale = 0.125f;        // 1 / sqrt(64), exact in fp32
constexpr float kLog2e = 1.4426950408889634f;

// Device error codes written into the error word (first writer wins).
constexpr unsigned kDevErrTimeout = 1u;
constexpr unsigned kDevErrBounds = 2u;

// Everything a kernel needs about one call.
struct Problem {
  const float* q;   // [C][32][64]
  const float* k;   // [P+C][8][64]
  const float* v;   // [P+C][8][64]
  float* out;       // [C][32][64]
  int C;            // chunk rows
  int P;            // cached prefix length
  unsigned* err;    // device error word
};

__device__ __forceinline__ void record_error(unsigned* err, unsigned code) {
  atomicCAS(err, 0u, code);
}

// Visible keys of chunk rows [t0, t0 + rows) clipped to the chunk: the unit's
// key range is [0, P + min(t0 + rows, C)).
__host__ __device__ __forceinline__ int unit_keys(int P, int C, int t0, int rows) {
  const int end = t0 + rows < C ? t0 + rows : C;
  return P + end;
}

// Host launchers, one per kernel family (defined in their own .cu files).
cudaError_t launch_reference(const Problem& p, cudaStream_t stream);
cudaError_t launch_ffma(const Problem& p, cudaStream_t stream);
int launch_tc(const Problem& p, cudaStream_t stream);             // returns an ATTN_* code
int launch_tc_fault_test(const Problem& p, cudaStream_t stream);  // skips a load, 20 ms waits
// Decode (decode.cu): how many split blocks the current device holds at once
// (first call per device sets the kernel up); split count and segment length
// for B sequences of at most max_context keys; workspace bytes for the
// partials; launch. The int results are ATTN_* codes.
int decode_slots(int* slots);
int decode_splits(int B, int max_context, int splits_hint, int slots, int* split_len);
size_t decode_workspace_bytes(int B, int splits);
// fault != 0 (failure-path test): the first tile of every block is never
// loaded and every wait is limited to 20 ms (2 s otherwise).
int launch_decode(const float* q, const float* k_pages, const float* v_pages, const int* table,
                  const int* ctx_lens, float* out, float* parts, int B, int max_blocks, int num_pages,
                  int max_context, int split_len, int splits, unsigned* err, cudaStream_t stream, int fault = 0);
// Three-kernel score-matrix attention (naive.cu): workspace bytes, the row
// limit of its grids, and one launcher per kernel.
size_t naive_workspace_bytes(int C, int P);
int naive_max_rows();
cudaError_t launch_naive_scores(const float* q, const float* k, float* S, int C, int P, cudaStream_t stream);
cudaError_t launch_naive_softmax(float* S, int C, int P, cudaStream_t stream);
cudaError_t launch_naive_weighted_sum(const float* S, const float* v, float* out, int C, int P,
                                      cudaStream_t stream);
// The fixed partials scratch of attn_decode_paged_noalloc (decode.cu) and its
// device address on the current device (looked up on the first call).
constexpr size_t kDecodeScratchBytes = size_t(4) << 20;
cudaError_t decode_scratch(float** ptr);
// BF16 K/V cache (tc_bf16.cu): p.k / p.v point at [P + C][8][64] bf16 caches.
int launch_tc_bf16(const Problem& p, cudaStream_t stream);
// fp32 K/V cache through the same kernel, K/V split into bf16 pairs in place.
int launch_tc_bf16x3(const Problem& p, cudaStream_t stream);
// Paged K/V: p.k / p.v point at [num_pages * 16][8][64] page pools.
int launch_tc_paged(const Problem& p, const int* table, int num_pages, cudaStream_t stream);

// Tensor-pipe rate measurement (peak.cu): `ctas` CTAs each issue `iters`
// dense M = 128, N = n MMAs (kind::tf32, or kind::f16 with bf16 operands).
int launch_tensor_peak(int bf16, int n, int iters, int ctas, unsigned* err, cudaStream_t stream);

}  // namespace attn
