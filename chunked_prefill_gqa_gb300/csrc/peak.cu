// peak.cu -- a measurement of the tensor pipe, not part of the attention
// method: every SM issues dense tcgen05.mma instructions back to back into
// tensor memory, so the time of a launch gives the rate the prefill kernels'
// contractions are held against. Page 1 ("Inference Attention 2: Flash
// Prefill Against a Cached Prefix", What you will learn) has the reader decide
// from SM throughput whether a kernel is compute-bound; for the split-TF32
// kernel that needs the kind::tf32 rate of this GPU, which no library GEMM
// reports.
//
// One CTA per SM (its dynamic shared memory leaves room for no second one),
// 128 threads. The operands are 128-byte-swizzled K-major tiles in shared
// memory filled with pseudo-random values in [-0.5, 0.5) (operand values
// change the power drawn, and so the clock): A is 128 rows, B is N rows, each
// row one 128-byte swizzle row, so one MMA of K = 8 (tf32) or 16 (bf16)
// elements reads 32 bytes of every row. Thread 0 issues `iters` MMAs of M =
// 128, N = n, alternating between two accumulators, commits once and waits
// (bounded) for completion; an expired wait records ATTN_ETIMEOUT.
#include "common.cuh"
#include "tc_ptx.cuh"

namespace attn {
namespace {

using namespace tc;

constexpr int kPeakThreads = 128;
constexpr uint32_t kPeakA = 0;              // 128 rows x 128 B
constexpr uint32_t kPeakB = 128 * 128;      // up to 256 rows x 128 B
constexpr uint32_t kPeakBar = kPeakB + 256 * 128;
constexpr uint32_t kPeakSmem = 120 * 1024;  // > half an SM's shared memory: one CTA per SM

__device__ __forceinline__ uint32_t mix32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

template <int kBf16>
__global__ void __launch_bounds__(kPeakThreads, 1)
tensor_peak_kernel(int n, int iters, unsigned long long timeout_ns, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* done = reinterpret_cast<uint64_t*>(smem + kPeakBar);
  uint32_t* holder = reinterpret_cast<uint32_t*>(smem + kPeakBar + 8);

  // Operand values: [-0.5, 0.5) as fp32, or two such bf16 per word.
  uint32_t* words = reinterpret_cast<uint32_t*>(smem);
  for (uint32_t i = threadIdx.x; i < kPeakBar / 4; i += kPeakThreads) {
    const uint32_t h = mix32(i * 0x9e3779b9u + blockIdx.x);
    const float a = __uint_as_float(0x3F800000u | (h >> 9)) - 1.5f;
    if constexpr (kBf16) {
      const float b = __uint_as_float(0x3F800000u | (mix32(h) >> 9)) - 1.5f;
      words[i] = pack_bf16_rn(a, b);
    } else {
      words[i] = __float_as_uint(a);
    }
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (threadIdx.x < 32) {
    tmem_alloc(holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;

  if (threadIdx.x == 0) {
    const uint32_t a = smem_u32(smem + kPeakA), b = smem_u32(smem + kPeakB);
    const uint32_t idesc = kBf16 ? idesc_bf16(128, n, false) : idesc_tf32(128, n);
#pragma unroll 1
    for (int i = 0; i < iters; ++i) {
      const uint32_t d = tmem + (uint32_t)(i & 1) * 256u;
      const uint64_t ad = sdesc_sw128(a + (i & 3) * 32), bd = sdesc_sw128(b + (i & 3) * 32);
      if constexpr (kBf16)
        mma_f16_ss(d, ad, bd, idesc, i >= 2);
      else
        mma_tf32_ss(d, ad, bd, idesc, i >= 2);
    }
    mma_commit(done);
    if (!mbar_wait(done, 0, timeout_ns)) record_error(err, kDevErrTimeout);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) tmem_dealloc(tmem, 512);
}

}  // namespace

int launch_tensor_peak(int bf16, int n, int iters, int ctas, unsigned* err, cudaStream_t stream) {
  static_assert(kPeakBar + 16 + 1024 <= kPeakSmem, "operands exceed the dynamic shared memory");
  const void* fn = bf16 ? (const void*)tensor_peak_kernel<1> : (const void*)tensor_peak_kernel<0>;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPeakSmem) != cudaSuccess)
    return ATTN_ECUDA;
  if (bf16)
    tensor_peak_kernel<1><<<ctas, kPeakThreads, kPeakSmem, stream>>>(n, iters, 2000000000ull, err);
  else
    tensor_peak_kernel<0><<<ctas, kPeakThreads, kPeakSmem, stream>>>(n, iters, 2000000000ull, err);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ELAUNCH;
}

}  // namespace attn
