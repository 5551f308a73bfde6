// ffma.cu -- flash prefill on the FP32 CUDA cores (exact fp32 products).
//
// The tiled algorithm of "Inference Attention 2: Flash Prefill Against a
// Cached Prefix" (Lesson): a tile of query rows stays resident, each K/V
// tile is staged in shared memory once and consumed by every resident row,
// and m, l and the accumulator are carried across tiles with the rescale by
// exp(m_old - m_new) and the division by l at the end (one reciprocal per
// row). GQA packing ("FlashAttention and inference kernels", GQA read
// amplification): a block owns 16 chunk positions x the 4 query heads of one
// KV head = 64 rows, so one K/V tile feeds all four heads. Causal skipping: the block loads keys [0, P + last
// row] only and masks elementwise only on tiles that cross the diagonal
// (same page, "How FlashAttention evolved", the causal mask).
//
// Block: 128 threads. Thread (rg, kg) = (tid / 16, tid % 16) owns rows
// 8 rg .. 8 rg + 7 and, for the scores, keys kg + 16 c (c = 0..3); for the
// output, head dimensions 4 kg .. 4 kg + 3. Row reductions run over the 16
// lanes that share rg. K and V tiles arrive by cp.async into a two-stage
// ring; the probabilities go through shared memory, transposed, to the PV
// product.
#include <mutex>

#include "common.cuh"

namespace attn {
namespace {

constexpr int kBq = 16;                 // chunk positions per block
constexpr int kM = kBq * kGroup;        // 64 resident rows
constexpr int kBc = 64;                 // keys per K/V tile
constexpr int kThreads = 128;
constexpr int kLd = 68;                 // padded row length (floats) of every smem array
constexpr int kTileFloats = 64 * kLd;
constexpr size_t kSmemBytes = sizeof(float) * (size_t)(kTileFloats * 6);  // Qt, 2 K, 2 V, Pt

__device__ __forceinline__ void cp_async16(float* dst, const float* src, bool valid) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
  const int n = valid ? 16 : 0;  // n == 0 writes zeros and reads nothing
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(p) = make_float4(a, b, c, d);
}

// Stage keys [j0, j0 + 64) of KV head g; rows at or past T become zeros.
__device__ __forceinline__ void load_kv_tile(const Problem& p, int g, int j0, int T,
                                             float* ks, float* vs, int tid) {
#pragma unroll
  for (int it = 0; it < (kBc * kD / 4) / kThreads; ++it) {
    const int idx = tid + it * kThreads;
    const int key = idx >> 4, c4 = idx & 15;
    const bool valid = j0 + key < T;
    const size_t src = ((size_t)(valid ? j0 + key : 0) * kHKV + g) * kD + c4 * 4;
    cp_async16(ks + key * kLd + c4 * 4, p.k + src, valid);
    cp_async16(vs + key * kLd + c4 * 4, p.v + src, valid);
  }
}

__global__ void __launch_bounds__(kThreads, 2)
ffma_kernel(Problem p, int n_qtiles) {
  extern __shared__ __align__(16) float smem[];
  float* Qt = smem;                        // [d][row], q * 1/8
  float* Ks = smem + kTileFloats;          // [2][key][d]
  float* Vs = smem + 3 * kTileFloats;      // [2][key][d]
  float* Pt = smem + 5 * kTileFloats;      // [key][row]

  // Longest units first: the last q-tiles see the most keys.
  const int qt = n_qtiles - 1 - (int)(blockIdx.x / kHKV);
  const int g = (int)(blockIdx.x % kHKV);
  const int t0 = qt * kBq;
  const int tid = threadIdx.x;
  const int kg = tid & 15, rg = tid >> 4;
  const int T = p.P + p.C;
  const int nkeys = unit_keys(p.P, p.C, t0, kBq);
  const int ntiles = (nkeys + kBc - 1) / kBc;

  // Resident query rows: row r = 4 * (position - t0) + (head - 4 g), scaled by 1/8.
#pragma unroll
  for (int it = 0; it < (kM * kD / 4) / kThreads; ++it) {
    const int idx = tid + it * kThreads;
    const int r = idx >> 4, c4 = idx & 15;
    const int pos = t0 + (r >> 2);
    float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
    if (pos < p.C) val = ld4(p.q + ((size_t)pos * kHQ + g * kGroup + (r & 3)) * kD + c4 * 4);
    Qt[(c4 * 4 + 0) * kLd + r] = val.x * kScale;
    Qt[(c4 * 4 + 1) * kLd + r] = val.y * kScale;
    Qt[(c4 * 4 + 2) * kLd + r] = val.z * kScale;
    Qt[(c4 * 4 + 3) * kLd + r] = val.w * kScale;
  }

  float o[8][4];
  float m[8], l[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    m[r] = -INFINITY;
    l[r] = 0.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) o[r][c] = 0.f;
  }

  load_kv_tile(p, g, 0, T, Ks, Vs, tid);
  cp_async_commit();

  for (int it = 0; it < ntiles; ++it) {
    const int buf = it & 1;
    const int j0 = it * kBc;
    if (it + 1 < ntiles) {
      load_kv_tile(p, g, j0 + kBc, T, Ks + (buf ^ 1) * kTileFloats, Vs + (buf ^ 1) * kTileFloats, tid);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    const float* kb = Ks + buf * kTileFloats;
    const float* vb = Vs + buf * kTileFloats;

    // S = (Q / 8) K^T for rows 8 rg.. and keys kg + 16 c.
    float s[8][4];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) s[r][c] = 0.f;
#pragma unroll 2
    for (int d4 = 0; d4 < kD / 4; ++d4) {
      float4 kk[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) kk[c] = ld4(kb + (kg + 16 * c) * kLd + d4 * 4);
#pragma unroll
      for (int dd = 0; dd < 4; ++dd) {
        const float* qp = Qt + (d4 * 4 + dd) * kLd + rg * 8;
        const float4 qa = ld4(qp), qb = ld4(qp + 4);
        const float qv[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float kd = dd == 0 ? kk[c].x : dd == 1 ? kk[c].y : dd == 2 ? kk[c].z : kk[c].w;
#pragma unroll
          for (int r = 0; r < 8; ++r) s[r][c] = fmaf(qv[r], kd, s[r][c]);
        }
      }
    }

    // Diagonal tiles only: key j is visible to position t iff j <= P + t.
    if (j0 + kBc - 1 > p.P + t0) {
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const int limit = p.P + t0 + ((rg * 8 + r) >> 2);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          if (j0 + kg + 16 * c > limit) s[r][c] = -INFINITY;
      }
    }

    // Online softmax update. l holds this thread's partial sum; every lane of a
    // row applies the same alpha, so the partials add up to l at the end.
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float mx = fmaxf(fmaxf(s[r][0], s[r][1]), fmaxf(s[r][2], s[r][3]));
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mnew = fmaxf(m[r], mx);
      const float mref = mnew == -INFINITY ? 0.f : mnew;  // fully masked so far: no NaN
      // e^(s - m) = 2^(s log2(e) - m log2(e)): one FFMA and one ex2.
      const float alpha = ex2((m[r] - mref) * kLog2e);
      const float mc = mref * kLog2e;
      float lsum = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float pj = ex2(fmaf(s[r][c], kLog2e, -mc));
        s[r][c] = pj;
        lsum += pj;
      }
      l[r] = fmaf(l[r], alpha, lsum);
#pragma unroll
      for (int c = 0; c < 4; ++c) o[r][c] *= alpha;
      m[r] = mnew;
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      float* pp = Pt + (kg + 16 * c) * kLd + rg * 8;
      st4(pp, s[0][c], s[1][c], s[2][c], s[3][c]);
      st4(pp + 4, s[4][c], s[5][c], s[6][c], s[7][c]);
    }
    __syncthreads();

    // O += P V for rows 8 rg.. and head dimensions 4 kg..
#pragma unroll 4
    for (int j = 0; j < kBc; ++j) {
      const float* pp = Pt + j * kLd + rg * 8;
      const float4 pa = ld4(pp), pb = ld4(pp + 4);
      const float pv[8] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
      const float4 vv = ld4(vb + j * kLd + kg * 4);
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        o[r][0] = fmaf(pv[r], vv.x, o[r][0]);
        o[r][1] = fmaf(pv[r], vv.y, o[r][1]);
        o[r][2] = fmaf(pv[r], vv.z, o[r][2]);
        o[r][3] = fmaf(pv[r], vv.w, o[r][3]);
      }
    }
    __syncthreads();
  }

  // Normalise by l at the very end: one reciprocal per row.
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    float lr = l[r];
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) lr += __shfl_xor_sync(0xffffffffu, lr, off);
    const int row = rg * 8 + r;
    const int pos = t0 + (row >> 2);
    if (pos < p.C) {
      float* dst = p.out + ((size_t)pos * kHQ + g * kGroup + (row & 3)) * kD + kg * 4;
      const float inv = 1.f / lr;
      st4(dst, o[r][0] * inv, o[r][1] * inv, o[r][2] * inv, o[r][3] * inv);
    }
  }
}

}  // namespace

cudaError_t launch_ffma(const Problem& p, cudaStream_t stream) {
  static bool configured[64] = {};  // the attribute is set once per device
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!configured[dev]) {
    e = cudaFuncSetAttribute(ffma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  const int n_qtiles = (p.C + kBq - 1) / kBq;
  ffma_kernel<<<n_qtiles * kHKV, kThreads, kSmemBytes, stream>>>(p, n_qtiles);
  return cudaGetLastError();
}

}  // namespace attn
