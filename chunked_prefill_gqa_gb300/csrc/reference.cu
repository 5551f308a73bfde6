// reference.cu -- the in-run timing reference: the untiled design the page
// "Inference Attention 2: Flash Prefill Against a Cached Prefix" (Starter
// code) times its lab against, rebuilt from its description.
//
// The design in prose: every (chunk row, query head) is an independent task
// for one warp; the task walks its whole visible prefix, key by key, loading
// each key and value row straight from global memory (nothing is staged or
// shared between tasks, so a K/V row is fetched once per query row and head
// that sees it), and folds each key into a running maximum, denominator and
// accumulator with the online rescale at every key. Correct, and slow on
// purpose: it is the per-row re-reading the tiled kernels remove.
//
// Mapping used here: a flat grid of tasks ordered head-major (task = h * C +
// i), so the warps of a block take consecutive rows of one head; lane l holds
// head dimensions 2l and 2l + 1 of the query, the accumulator and the output.
// Scores are carried in log2 units (s * log2(e) / 8), so every exponential
// is a single exp2.
#include "common.cuh"

namespace attn {
namespace {

constexpr int kTaskWarps = 4;  // tasks (warps) per block

__device__ __forceinline__ float warp_total(float x) {
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
  return x;
}

__global__ void __launch_bounds__(kTaskWarps * 32)
reference_kernel(Problem p) {
  const long long task = (long long)blockIdx.x * kTaskWarps + (threadIdx.x >> 5);
  if (task >= (long long)p.C * kHQ) return;
  const int h = (int)(task / p.C);
  const int i = (int)(task % p.C);
  const int lane = threadIdx.x & 31;

  // Row-major [pos][head][64] tensors read as float2: dims (2 lane, 2 lane + 1).
  constexpr int kPosStride = kHKV * kD / 2;  // float2 elements between positions
  const float2 qd = reinterpret_cast<const float2*>(p.q + ((size_t)i * kHQ + h) * kD)[lane];
  const float2* kcol = reinterpret_cast<const float2*>(p.k + (size_t)(h / kGroup) * kD) + lane;
  const float2* vcol = reinterpret_cast<const float2*>(p.v + (size_t)(h / kGroup) * kD) + lane;
  const float to_log2 = kScale * kLog2e;

  float run_max = -INFINITY;  // log2 units
  float denom = 0.f;
  float2 acc = make_float2(0.f, 0.f);
  const int visible = p.P + i + 1;  // keys 0 .. P + i
  for (int j = 0; j < visible; ++j) {
    const float2 kj = kcol[(size_t)j * kPosStride];
    const float t = warp_total(fmaf(qd.x, kj.x, qd.y * kj.y)) * to_log2;
    const float top = fmaxf(run_max, t);
    const float keep = exp2f(run_max - top);  // 0 at the first key
    const float w = exp2f(t - top);
    const float2 vj = vcol[(size_t)j * kPosStride];
    denom = fmaf(denom, keep, w);
    acc.x = fmaf(acc.x, keep, w * vj.x);
    acc.y = fmaf(acc.y, keep, w * vj.y);
    run_max = top;
  }
  reinterpret_cast<float2*>(p.out + ((size_t)i * kHQ + h) * kD)[lane] = make_float2(acc.x / denom, acc.y / denom);
}

}  // namespace

cudaError_t launch_reference(const Problem& p, cudaStream_t stream) {
  const long long tasks = (long long)p.C * kHQ;
  const unsigned blocks = (unsigned)((tasks + kTaskWarps - 1) / kTaskWarps);
  reference_kernel<<<blocks, kTaskWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace attn
