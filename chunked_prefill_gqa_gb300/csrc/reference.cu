// reference.cu -- the in-run timing reference: the starter design of
// "Inference Attention 2: Flash Prefill Against a Cached Prefix" (Starter
// code), rebuilt. One warp owns one (chunk row, query head) at a time; its 32
// lanes hold the 64 query elements two apiece, every key is read straight
// from global memory, the dot product is reduced across the warp, and the
// running maximum, denominator and accumulator are rescaled at every key.
// Each row walks its whole prefix alone, which is the cost the page measures
// the tiled kernels against. Correct, online and deliberately untiled.
#include "common.cuh"

namespace attn {
namespace {

constexpr int kRowsPerBlock = 64;     // chunk rows per block
constexpr int kWarps = 8;             // each warp takes 8 consecutive rows

__global__ void __launch_bounds__(kWarps * 32)
reference_kernel(Problem p) {
  const int head = blockIdx.y;
  const int kvh = head / kGroup;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int first = blockIdx.x * kRowsPerBlock + warp * (kRowsPerBlock / kWarps);
  for (int r = 0; r < kRowsPerBlock / kWarps; ++r) {
    const int row = first + r;
    if (row >= p.C) return;
    const float* qrow = p.q + ((size_t)row * kHQ + head) * kD;
    const float qlo = qrow[lane];
    const float qhi = qrow[lane + 32];
    float m = -INFINITY, l = 0.f, olo = 0.f, ohi = 0.f;
    const int last = p.P + row;  // row i sees keys j <= P + i
    for (int j = 0; j <= last; ++j) {
      const size_t base = ((size_t)j * kHKV + kvh) * kD;
      float dot = fmaf(qlo, p.k[base + lane], qhi * p.k[base + lane + 32]);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
      const float s = dot * kScale;
      const float mnew = fmaxf(m, s);
      const float alpha = expf(m - mnew);   // 0 at the first key (m = -inf)
      const float pj = expf(s - mnew);
      l = fmaf(l, alpha, pj);
      olo = fmaf(olo, alpha, pj * p.v[base + lane]);
      ohi = fmaf(ohi, alpha, pj * p.v[base + lane + 32]);
      m = mnew;
    }
    float* orow = p.out + ((size_t)row * kHQ + head) * kD;
    orow[lane] = olo / l;
    orow[lane + 32] = ohi / l;
  }
}

}  // namespace

cudaError_t launch_reference(const Problem& p, cudaStream_t stream) {
  dim3 grid((p.C + kRowsPerBlock - 1) / kRowsPerBlock, kHQ);
  reference_kernel<<<grid, kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace attn
