// naive.cu -- the three-kernel attention of an eager framework, with the whole
// score matrix in global memory ("Inference Attention 1: The Full Score
// Matrix", Lesson): a scores matmul, an in-place row softmax and a weighted
// sum. It is kept as the in-run measurement of what that matrix costs next to
// the flash kernels, which never form it.
//
// Workspace: S [32][C][P + C] fp32, head-major, row i of head h at
// S + (h C + i)(P + C). For the chunk rows i at positions P + i the scores
// kernel writes q.k / 8 for keys j <= P + i and -inf above the diagonal; the
// softmax replaces every row by its probabilities (0 above the diagonal); the
// weighted sum multiplies them by V. With P = 0 this is exactly the page's
// full prompt (T x T per head).
#include "common.cuh"

namespace attn {
namespace {

constexpr int kTile = 64;     // rows x keys of a scores tile; rows x head dims of an output tile
constexpr int kKeys = 32;     // keys per staged tile of the weighted sum
constexpr int kThreads = 256;
constexpr int kPad = 68;      // padded smem row (floats)

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// Scores: block (key tile, row tile, head). Thread (ty, tx) = (tid / 16,
// tid % 16) owns rows 4 ty .. 4 ty + 3 and keys 4 tx .. 4 tx + 3 of the tile.
__global__ void __launch_bounds__(kThreads)
naive_scores_kernel(const float* __restrict__ q, const float* __restrict__ k, float* __restrict__ S, int C,
                    int P) {
  __shared__ __align__(16) float Qs[kD][kPad];  // [d][row], q / 8
  __shared__ __align__(16) float Ks[kD][kPad];  // [d][key]
  const int T = P + C;
  const int j0 = blockIdx.x * kTile, r0 = blockIdx.y * kTile, h = blockIdx.z;
  const int g = h / kGroup;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int last_row = min(r0 + kTile, C) - 1;
  const bool vec = (T & 3) == 0;
  float acc[4][4];

  if (j0 > P + last_row) {  // the whole tile lies above the diagonal
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] = -INFINITY;
  } else {
#pragma unroll
    for (int it = 0; it < (kTile * kD / 4) / kThreads; ++it) {
      const int idx = tid + it * kThreads;
      const int row = idx >> 4, c4 = idx & 15;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
      if (r0 + row < C) a = ld4(q + ((size_t)(r0 + row) * kHQ + h) * kD + c4 * 4);
      if (j0 + row < T) b = ld4(k + ((size_t)(j0 + row) * kHKV + g) * kD + c4 * 4);
      Qs[c4 * 4 + 0][row] = a.x * kScale;
      Qs[c4 * 4 + 1][row] = a.y * kScale;
      Qs[c4 * 4 + 2][row] = a.z * kScale;
      Qs[c4 * 4 + 3][row] = a.w * kScale;
      Ks[c4 * 4 + 0][row] = b.x;
      Ks[c4 * 4 + 1][row] = b.y;
      Ks[c4 * 4 + 2][row] = b.z;
      Ks[c4 * 4 + 3][row] = b.w;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
#pragma unroll 8
    for (int d = 0; d < kD; ++d) {
      const float4 a = ld4(&Qs[d][4 * ty]);
      const float4 b = ld4(&Ks[d][4 * tx]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
    }
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (j0 + 4 * tx + c > P + r0 + 4 * ty + r) acc[r][c] = -INFINITY;  // causal mask
  }

#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = r0 + 4 * ty + r;
    const int j = j0 + 4 * tx;
    if (i >= C) continue;
    float* dst = S + ((size_t)h * C + i) * T + j;
    if (vec && j + 3 < T) {
      *reinterpret_cast<float4*>(dst) = make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (j + c < T) dst[c] = acc[r][c];
    }
  }
}

// Row softmax in place: one warp per row (head h, chunk row i). Pass 1 takes
// the maximum of the visible scores, pass 2 sums e^(s - m), pass 3 writes the
// probabilities and zeros above the diagonal.
__global__ void __launch_bounds__(kThreads)
naive_softmax_kernel(float* __restrict__ S, int C, int P) {
  const int T = P + C;
  const long long row = (long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= 32LL * C) return;
  const int i = (int)(row % C);
  float* s = S + (size_t)row * T;
  const int vis = P + i + 1;

  float m = -INFINITY;
  for (int j = lane; j < vis; j += 32) m = fmaxf(m, s[j]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float l = 0.f;
  for (int j = lane; j < vis; j += 32) l += exp2f((s[j] - m) * kLog2e);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  const float inv = 1.f / l;
  for (int j = lane; j < vis; j += 32) s[j] = exp2f((s[j] - m) * kLog2e) * inv;
  for (int j = vis + lane; j < T; j += 32) s[j] = 0.f;
}

// Weighted sum: block (row tile, head), longest row tiles first. Thread
// (ty, tx) owns rows 4 ty .. 4 ty + 3 and head dims 4 tx .. 4 tx + 3; keys are
// staged 32 at a time, the probabilities transposed to [key][row].
__global__ void __launch_bounds__(kThreads)
naive_weighted_sum_kernel(const float* __restrict__ S, const float* __restrict__ v, float* __restrict__ out,
                          int C, int P) {
  __shared__ __align__(16) float Ps[kKeys][kPad];  // [key][row]
  __shared__ __align__(16) float Vs[kKeys][kD];    // [key][d]
  const int T = P + C;
  const int r0 = (gridDim.x - 1 - blockIdx.x) * kTile, h = blockIdx.y;
  const int g = h / kGroup;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int nkeys = P + min(r0 + kTile, C);  // keys visible to the tile's last row
  float acc[4][4] = {};

  for (int k0 = 0; k0 < nkeys; k0 += kKeys) {
    // probabilities: 64 rows x 32 keys, one float per thread per step
#pragma unroll
    for (int it = 0; it < (kTile * kKeys) / kThreads; ++it) {
      const int idx = tid + it * kThreads;
      const int row = idx >> 5, key = idx & 31;
      const int i = r0 + row, j = k0 + key;
      Ps[key][row] = (i < C && j < T) ? S[((size_t)h * C + i) * T + j] : 0.f;
    }
#pragma unroll
    for (int it = 0; it < (kKeys * kD / 4) / kThreads; ++it) {
      const int idx = tid + it * kThreads;
      const int key = idx >> 4, c4 = idx & 15;
      float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
      if (k0 + key < T) b = ld4(v + ((size_t)(k0 + key) * kHKV + g) * kD + c4 * 4);
      *reinterpret_cast<float4*>(&Vs[key][c4 * 4]) = b;
    }
    __syncthreads();
#pragma unroll 8
    for (int key = 0; key < kKeys; ++key) {
      const float4 a = ld4(&Ps[key][4 * ty]);
      const float4 b = ld4(&Vs[key][4 * tx]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
    }
    __syncthreads();
  }

#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int i = r0 + 4 * ty + r;
    if (i < C)
      *reinterpret_cast<float4*>(out + ((size_t)i * kHQ + h) * kD + 4 * tx) =
          make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
  }
}

}  // namespace

size_t naive_workspace_bytes(int C, int P) { return (size_t)kHQ * C * ((size_t)P + C) * sizeof(float); }

int naive_max_rows() { return 65535 * kTile; }

cudaError_t launch_naive_scores(const float* q, const float* k, float* S, int C, int P, cudaStream_t stream) {
  const int T = P + C;
  naive_scores_kernel<<<dim3((T + kTile - 1) / kTile, (C + kTile - 1) / kTile, kHQ), kThreads, 0, stream>>>(
      q, k, S, C, P);
  return cudaGetLastError();
}

cudaError_t launch_naive_softmax(float* S, int C, int P, cudaStream_t stream) {
  const long long rows = 32LL * C;
  const int per = kThreads / 32;
  naive_softmax_kernel<<<(unsigned)((rows + per - 1) / per), kThreads, 0, stream>>>(S, C, P);
  return cudaGetLastError();
}

cudaError_t launch_naive_weighted_sum(const float* S, const float* v, float* out, int C, int P,
                                      cudaStream_t stream) {
  naive_weighted_sum_kernel<<<dim3((C + kTile - 1) / kTile, kHQ), kThreads, 0, stream>>>(S, v, out, C, P);
  return cudaGetLastError();
}

}  // namespace attn
