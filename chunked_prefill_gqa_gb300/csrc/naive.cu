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
#include <mutex>

#include "common.cuh"

namespace attn {
namespace {

constexpr int kRows = 128;    // rows of a scores or weighted-sum block tile
constexpr int kCols = 64;     // keys of a scores tile; head dims of a weighted-sum tile
constexpr int kKeys = 32;     // keys per staged chunk of the weighted sum
constexpr int kThreads = 256; // thread (ty, tx) = (tid / 16, tid % 16): rows 8 ty .. 8 ty + 7, columns 4 tx .. 4 tx + 3
constexpr int kLdR = kRows + 4;  // padded smem row (floats) of a [.][row] array

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

// 8 x 4 register tile update: acc[r][c] += a[r] b[c].
__device__ __forceinline__ void fma8x4(float (&acc)[8][4], const float4 a0, const float4 a1, const float4 b) {
  const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
  for (int r = 0; r < 8; ++r)
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
}

// Scores: block (64-key tile, 128-row tile, head). q / 8 and K staged
// transposed ([d][row], [d][key]); tiles wholly above the diagonal are written
// as -inf without computing.
__global__ void __launch_bounds__(kThreads)
naive_scores_kernel(const float* __restrict__ q, const float* __restrict__ k, float* __restrict__ S, int C,
                    int P) {
  extern __shared__ __align__(16) float dsm[];
  float (*Qs)[kLdR] = reinterpret_cast<float (*)[kLdR]>(dsm);                      // [d][row]
  float (*Ks)[kCols + 4] = reinterpret_cast<float (*)[kCols + 4]>(dsm + kD * kLdR);  // [d][key]
  const int T = P + C;
  const int j0 = blockIdx.x * kCols, r0 = blockIdx.y * kRows, h = blockIdx.z;
  const int g = h / kGroup;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int last_row = min(r0 + kRows, C) - 1;
  const bool vec = (T & 3) == 0;
  float acc[8][4];

  if (j0 > P + last_row) {  // the whole tile lies above the diagonal
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] = -INFINITY;
  } else {
    // q rows: 128 x 64 floats, 8 float4 per thread; K rows: 64 x 64, 4 per thread.
#pragma unroll
    for (int it = 0; it < (kRows * kD / 4) / kThreads; ++it) {
      const int idx = tid + it * kThreads;
      const int row = idx >> 4, c4 = idx & 15;
      float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
      if (r0 + row < C) a = ld4(q + ((size_t)(r0 + row) * kHQ + h) * kD + c4 * 4);
      Qs[c4 * 4 + 0][row] = a.x * kScale;
      Qs[c4 * 4 + 1][row] = a.y * kScale;
      Qs[c4 * 4 + 2][row] = a.z * kScale;
      Qs[c4 * 4 + 3][row] = a.w * kScale;
    }
#pragma unroll
    for (int it = 0; it < (kCols * kD / 4) / kThreads; ++it) {
      const int idx = tid + it * kThreads;
      const int row = idx >> 4, c4 = idx & 15;
      float4 b = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j0 + row < T) b = ld4(k + ((size_t)(j0 + row) * kHKV + g) * kD + c4 * 4);
      Ks[c4 * 4 + 0][row] = b.x;
      Ks[c4 * 4 + 1][row] = b.y;
      Ks[c4 * 4 + 2][row] = b.z;
      Ks[c4 * 4 + 3][row] = b.w;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] = 0.f;
#pragma unroll 8
    for (int d = 0; d < kD; ++d)
      fma8x4(acc, ld4(&Qs[d][8 * ty]), ld4(&Qs[d][8 * ty + 4]), ld4(&Ks[d][4 * tx]));
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        if (j0 + 4 * tx + c > P + r0 + 8 * ty + r) acc[r][c] = -INFINITY;  // causal mask
  }

#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int i = r0 + 8 * ty + r;
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

// Weighted sum: block (128-row tile, head), longest row tiles first. Keys in
// chunks of 32: the probabilities staged transposed ([key][row]) and V
// ([key][d]); the next chunk's global loads are in registers while the current
// one is used. Keys past the tile's last visible key are never read.
__global__ void __launch_bounds__(kThreads)
naive_weighted_sum_kernel(const float* __restrict__ S, const float* __restrict__ v, float* __restrict__ out,
                          int C, int P) {
  extern __shared__ __align__(16) float dsm[];
  float (*Ps)[kKeys][kLdR] = reinterpret_cast<float (*)[kKeys][kLdR]>(dsm);                 // [buffer][key][row]
  float (*Vs)[kKeys][kD] = reinterpret_cast<float (*)[kKeys][kD]>(dsm + 2 * kKeys * kLdR);  // [buffer][key][d]
  const int T = P + C;
  const int r0 = (gridDim.x - 1 - blockIdx.x) * kRows, h = blockIdx.y;
  const int g = h / kGroup;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int nkeys = P + min(r0 + kRows, C);  // keys visible to the tile's last row
  const int nchunks = (nkeys + kKeys - 1) / kKeys;
  float acc[8][4] = {};

  // A chunk: 128 rows x 32 keys of S (16 per thread, a warp reads one row's 32
  // keys) and 32 keys x 64 dims of V (2 float4 per thread).
  float pr[(kRows * kKeys) / kThreads];
  float4 vr[(kKeys * kD / 4) / kThreads];
  auto fetch = [&](int k0) {
#pragma unroll
    for (int it = 0; it < (kRows * kKeys) / kThreads; ++it) {
      const int idx = tid + it * kThreads;
      const int row = idx >> 5, key = idx & 31;
      const int i = r0 + row, j = k0 + key;
      pr[it] = (i < C && j < T) ? __ldg(S + ((size_t)h * C + i) * T + j) : 0.f;
    }
#pragma unroll
    for (int it = 0; it < (kKeys * kD / 4) / kThreads; ++it) {
      const int idx = tid + it * kThreads;
      const int key = idx >> 4, c4 = idx & 15;
      vr[it] = (k0 + key < T) ? __ldg(reinterpret_cast<const float4*>(v + ((size_t)(k0 + key) * kHKV + g) * kD) + c4)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  };
  auto stash = [&](int buf) {
#pragma unroll
    for (int it = 0; it < (kRows * kKeys) / kThreads; ++it) {
      const int idx = tid + it * kThreads;
      Ps[buf][idx & 31][idx >> 5] = pr[it];
    }
#pragma unroll
    for (int it = 0; it < (kKeys * kD / 4) / kThreads; ++it) {
      const int idx = tid + it * kThreads;
      *reinterpret_cast<float4*>(&Vs[buf][idx >> 4][(idx & 15) * 4]) = vr[it];
    }
  };

  fetch(0);
  stash(0);
  __syncthreads();
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    if (c + 1 < nchunks) fetch((c + 1) * kKeys);
#pragma unroll 8
    for (int key = 0; key < kKeys; ++key)
      fma8x4(acc, ld4(&Ps[buf][key][8 * ty]), ld4(&Ps[buf][key][8 * ty + 4]), ld4(&Vs[buf][key][4 * tx]));
    if (c + 1 < nchunks) stash(buf ^ 1);  // the other buffer was last read before the previous barrier
    __syncthreads();
  }

#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int i = r0 + 8 * ty + r;
    if (i < C)
      *reinterpret_cast<float4*>(out + ((size_t)i * kHQ + h) * kD + 4 * tx) =
          make_float4(acc[r][0], acc[r][1], acc[r][2], acc[r][3]);
  }
}

constexpr size_t kScoresSmem = sizeof(float) * (kD * kLdR + kD * (kCols + 4));   // 50,176 B
constexpr size_t kWsumSmem = sizeof(float) * (2 * kKeys * kLdR + 2 * kKeys * kD);  // 51,200 B

// Both tiled kernels use a little more than 48 KB of shared memory, which
// needs the per-kernel opt-in once per device.
cudaError_t configure_device() {
  static bool configured[64] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(naive_scores_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kScoresSmem);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(naive_weighted_sum_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kWsumSmem);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  return cudaSuccess;
}

}  // namespace

size_t naive_workspace_bytes(int C, int P) { return (size_t)kHQ * C * ((size_t)P + C) * sizeof(float); }

int naive_max_rows() { return 65535 * kRows; }

cudaError_t launch_naive_scores(const float* q, const float* k, float* S, int C, int P, cudaStream_t stream) {
  const int T = P + C;
  const cudaError_t e = configure_device();
  if (e != cudaSuccess) return e;
  naive_scores_kernel<<<dim3((T + kCols - 1) / kCols, (C + kRows - 1) / kRows, kHQ), kThreads, kScoresSmem,
                        stream>>>(q, k, S, C, P);
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
  const cudaError_t e = configure_device();
  if (e != cudaSuccess) return e;
  naive_weighted_sum_kernel<<<dim3((C + kRows - 1) / kRows, kHQ), kThreads, kWsumSmem, stream>>>(S, v, out, C, P);
  return cudaGetLastError();
}

}  // namespace attn
