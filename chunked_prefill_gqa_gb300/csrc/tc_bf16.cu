// tc_bf16.cu -- flash prefill on the sm_103a tensor cores with bf16 operands
// (tcgen05 kind::f16, TMEM accumulators, TMA staging), for a K/V cache held in
// bf16 or in fp32.
//
// The operation is the one of tc.cu (causal GQA attention of a chunk at
// positions P..P+C-1, scale 1/8, online softmax; "Inference Attention 2: Flash
// Prefill Against a Cached Prefix", Lesson). Every fp32 operand x is carried as
// two bf16 terms, x = x1 + x2 (16 significant bits together), and products
// accumulate in fp32 on the tensor cores:
//   bf16 cache ("FlashAttention and inference kernels", inference: the KV cache
//   in BF16): K and V are operands exactly as stored, so
//       S  = q1 K^T + q2 K^T                 (4 + 4 MMAs of 128 x 128 x 16)
//       O += p1 V   + p2 V                   (8 + 8 MMAs of 128 x 64 x 16)
//   fp32 cache: converter warps split each landed K/V tile in place into
//   [x1 | x2], and each product keeps three of its four terms,
//       S  = q1 k1^T + q1 k2^T + q2 k1^T     (3 x 4 MMAs of 128 x 128 x 16)
//       O' = p1 [v1 | v2] + p2 v1            (8 MMAs of 128 x 128 x 16 on the
//                                             stacked [v1 | v2] operand, then 8
//                                             of 128 x 64 x 16 into O'[:, :64])
//       O  = O'[:, :64] + O'[:, 64:]          (added in the epilogue)
//   dropping only x2 y2, below 2^-15 of |x y| (hi rounded to nearest: |x2| <=
//   2^-8 |x|; p1 truncated: |p2| < 2^-7 p); the kept terms carry the residual
//   of each split, at most 2^-9 |x2|.
// K is a K-major operand and V an MN-major one ([key][d] rows, 128-byte
// swizzle), so V needs no transpose. P and the accumulators live in TMEM; P
// (p1 | p2) overwrites the S columns it came from, two bf16 per 32-bit column.
// q1 | q2 is a TMEM operand with the bf16 cache and a shared-memory one with the
// fp32 cache, whose TMEM holds the 128-column O' instead.
//
// Work unit (as in tc.cu): 32 chunk positions x the 4 query heads of one KV
// head = 128 rows, one TMEM lane each. Keys come in tiles of 128; tiles past
// the unit's last visible key are never loaded; only diagonal tiles are masked.
//
// Warp roles:
//   0-7   softmax: warp w owns TMEM lanes 32 (w % 4) .. + 31 and keys
//         64 (w / 4) .. + 63 of every tile; the two warps of a row set exchange
//         partial maxima and sums through shared memory. They split q (into
//         TMEM, or shared memory with the fp32 cache), run the online softmax,
//         write p1/p2, rescale O when the reference maximum moves, and write the
//         output.
//   8     K producer, 9 V producer: TMA loads of whole tiles.
//   10    QK issuer (allocates TMEM): QK(n) once K(n) is ready and S buffer
//         n % 3 is free (PV(n-3) complete).
//   11    PV issuer: PV(n) once P(n) is written and V(n) is ready.
//   12-15 (fp32 cache) converters: 12-13 split K tiles, 14-15 V tiles, each
//         warp 64 keys; a lane owns one key and rewrites, in place, exactly
//         the two 128-byte rows it read.
// Three S buffers let QK run two tiles ahead of the softmax. Every wait is
// bounded; on expiry the kernel records ATTN_ETIMEOUT, winds down and frees TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace attn {
namespace {

using namespace tc;

constexpr int kBq = 32;           // chunk positions per unit
constexpr int kM = kBq * kGroup;  // 128 rows = TMEM lanes
constexpr int kBc = 128;          // keys per tile
constexpr int kNumS = 3;          // S / P buffers in TMEM

constexpr int kSoftmaxWarps = 8;
constexpr int kKProducerWarp = 8;
constexpr int kVProducerWarp = 9;
constexpr int kQkWarp = 10;
constexpr int kPvWarp = 11;
constexpr int kFirstConvWarp = 12;  // fp32 cache only
constexpr int kConvWarpsPerOperand = 2;
template <bool kF32>
constexpr int threads_of() {
  return 32 * (kF32 ? kFirstConvWarp + 2 * kConvWarpsPerOperand : kPvWarp + 1);
}

// TMEM columns (32-bit each). bf16 cache: q1 [0,32), q2 [32,64), three S
// buffers [64,448), O [448,512). fp32 cache (q in shared memory): three S
// buffers [0,384), O' = [p1 v1 + p2 v1 | p1 v2] [384,512).
constexpr uint32_t kColQhi = 0;   // 64 bf16 per row = 32 columns
constexpr uint32_t kColQlo = 32;
template <bool kF32>
__host__ __device__ constexpr uint32_t col_s() { return kF32 ? 0u : 64u; }  // 128-column S buffers; p1 | p2 overwrite them
template <bool kF32>
__host__ __device__ constexpr uint32_t col_o() { return kF32 ? 384u : 448u; }
constexpr uint32_t kTmemCols = 512;

// Shared memory (byte offsets from a 1024-aligned base). A bf16 operand tile
// is 128 keys x 64 values = 128 rows of 128 bytes in the 128-byte swizzle
// (16 KB). With an fp32 cache a stage is 32 KB: TMA lands d 0-31 and d 32-63
// as two such 16 KB regions, and the converters overwrite them with x1 and x2;
// q1 and q2 come first (two 16 KB K-major operands), then three K stages and two
// V stages. The bf16 cache has four stages of each.
constexpr uint32_t kOperandBytes = kBc * kD * 2;  // 16 KB
constexpr uint32_t kShareO = 128 * 256;          // split-unit share: O rows, then m and l
constexpr uint32_t kShareBytes = kShareO + 2 * 128 * 4;
template <bool kF32>
struct Layout {
  static constexpr int kKS = kF32 ? 3 : 4;  // K ring stages
  static constexpr int kVS = kF32 ? 2 : 4;  // V ring stages (an fp32 V stage is converted while up to two wait)
  static constexpr uint32_t kStageBytes = kF32 ? 2 * kOperandBytes : kOperandBytes;
  static constexpr uint32_t kSmemQ = 0;  // fp32 cache: q1 | q2, K-major bf16 operands of 16 KB each
  static constexpr uint32_t kSmemK = kSmemQ + (kF32 ? 2 * kOperandBytes : 0);
  static constexpr uint32_t kSmemV = kSmemK + kKS * kStageBytes;
  static constexpr uint32_t kSmemBar = kSmemV + kVS * kStageBytes;
  static constexpr uint32_t kNumBars = 3 * kKS + 3 * kVS + 9 + 1 + 2 + 4 + 2;
  static constexpr uint32_t kSmemRed = kSmemBar + kNumBars * 8 + 16;  // [2 tile parities][2 key halves][128 rows]
  static constexpr uint32_t kSmemLsum = kSmemRed + 2 * 2 * 128 * 4;   // [2 key halves][128 rows]
  static constexpr uint32_t kSmemTotal = kSmemLsum + 2 * 128 * 4;
  static constexpr uint32_t kSmemAlloc = kSmemTotal + 1024;
  static_assert(kSmemAlloc <= 232448, "exceeds the 227 KB per-block shared memory limit");
};

static_assert(kM == 128 && kD == 64 && kBc == 128, "the MMA shapes below assume 128 x 128 x 64");
static_assert(col_s<false>() + 3 * 128 <= col_o<false>() && col_o<false>() + kD <= kTmemCols, "TMEM layout");
static_assert(col_s<true>() + 3 * 128 <= col_o<true>() && col_o<true>() + 2 * kD <= kTmemCols, "TMEM layout");

constexpr uint32_t kIdescQK = idesc_bf16(128, 128, false);
constexpr uint32_t kIdescPV = idesc_bf16(128, 64, true);
constexpr uint32_t kIdescPV128 = idesc_bf16(128, 128, true);
constexpr float kStaleLog2 = 8.0f;  // see tc.cu: a stale reference maximum keeps p <= 2^8

struct Params {
  Problem p;
  int n_units;
  int n_qtiles;
  unsigned long long timeout_ns;
  int unit_base;  // tail kernel: pair p splits unit unit_base + p
};

struct Bars {
  uint64_t* kfull;   // [K stages] TMA K landed
  uint64_t* kconv;   // [K stages] K split into k1 | k2 (fp32 cache)
  uint64_t* vconv;   // [V stages] V split into v1 | v2 (fp32 cache)
  uint64_t* kempty;  // [K stages] QK done with the stage
  uint64_t* vfull;   // [V stages] TMA V landed
  uint64_t* vempty;  // [V stages] PV done with the stage
  uint64_t* sfull;   // [kNumS] S written (MMA commit)
  uint64_t* pfull;   // [kNumS] P written and O rescaled (softmax warps)
  uint64_t* odone;   // [kNumS] PV(n) complete, barrier n % 3
  uint64_t* qready;  // Q hi/lo in TMEM
  uint64_t* drain;   // [2] MMA issuers' drain on abort
  uint64_t* pair;    // [4] row-set exchanges of the softmax warps
  uint64_t* partner;   // tail kernel, rank 0: rank 1's share of the unit has landed (one arrival + bulk-copy bytes)
  uint64_t* slotfree;  // tail kernel, rank 1: rank 0's K ring is free for that share (256 remote arrivals)
};

template <bool kF32>
__device__ __forceinline__ Bars carve_bars(uint8_t* base) {
  uint64_t* b = reinterpret_cast<uint64_t*>(base + Layout<kF32>::kSmemBar);
  constexpr int kKS = Layout<kF32>::kKS, kVS = Layout<kF32>::kVS;
  Bars r;
  r.kfull = b; b += kKS;
  r.kconv = b; b += kKS;
  r.vconv = b; b += kVS;
  r.kempty = b; b += kKS;
  r.vfull = b; b += kVS;
  r.vempty = b; b += kVS;
  r.sfull = b; b += kNumS;
  r.pfull = b; b += kNumS;
  r.odone = b; b += kNumS;
  r.qready = b++;
  r.drain = b; b += 2;
  r.pair = b; b += 4;
  r.partner = b++;
  r.slotfree = b++;
  return r;
}

__device__ __forceinline__ int unit_index(int k, int cta, int grid) {
  return k * grid + ((k & 1) ? (grid - 1 - cta) : cta);
}

struct Unit {
  int t0, g, ntiles;
};
__device__ __forceinline__ Unit decode_unit(int u, const Params& prm) {
  Unit w;
  const int qt = prm.n_qtiles - 1 - u / kHKV;  // longest units first
  w.g = u % kHKV;
  w.t0 = qt * kBq;
  const int nkeys = unit_keys(prm.p.P, prm.p.C, w.t0, kBq);
  w.ntiles = (nkeys + kBc - 1) / kBc;
  return w;
}

// kSplit == 1: whole units in snake order. kSplit == 2: launched after that
// grid as clusters of two CTAs; pair p splits unit unit_base + p along its key
// tiles (rank 0 the first half, rank 1 the rest) and merges the two
// online-softmax partials through distributed shared memory. kSplit == 3, 4,
// 8: the same with clusters of three, four or eight CTAs, that share of the
// tiles each (small chunks).
template <int kSplit>
__device__ __forceinline__ int work_unit(int k, int cta, int grid, const Params& prm) {
  if constexpr (kSplit == 2) return k == 0 ? prm.unit_base + (cta >> 1) : prm.n_units;
  else if constexpr (kSplit == 4) return k == 0 ? prm.unit_base + (cta >> 2) : prm.n_units;
  else if constexpr (kSplit == 8) return k == 0 ? prm.unit_base + (cta >> 3) : prm.n_units;
  else if constexpr (kSplit == 3) return k == 0 ? prm.unit_base + cta / 3 : prm.n_units;
  else if constexpr (kSplit == 12) return k == 0 ? prm.unit_base + cta / 12 : prm.n_units;
  else return unit_index(k, cta, grid);
}
template <int kSplit>
__device__ __forceinline__ void unit_range(const Unit& w, uint32_t rank, int* jb, int* je) {
  if constexpr (kSplit == 2) {
    *jb = rank == 0 ? 0 : w.ntiles / 2;
    *je = rank == 0 ? w.ntiles / 2 : w.ntiles;
  } else if constexpr (kSplit == 3 || kSplit == 4 || kSplit == 8 || kSplit == 12) {
    *jb = (int)rank * w.ntiles / kSplit;
    *je = ((int)rank + 1) * w.ntiles / kSplit;
  } else {
    *jb = 0;
    *je = w.ntiles;
  }
}

__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const Params& prm,
                                         volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (globaltimer_ns() - t0 > prm.timeout_ns) {
      record_error(prm.p.err, kDevErrTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, const Params& prm,
                                              volatile int* abort_flag) {
  const bool ok = wait_bar(bar, parity, prm, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

// As wait_bar_warp, for a barrier the partner CTA arrives on: the wait
// acquires at cluster scope, so the partner's released writes are visible.
__device__ __forceinline__ bool wait_bar_cluster_warp(uint64_t* bar, uint32_t parity, const Params& prm,
                                                      volatile int* abort_flag) {
  bool ok = mbar_try_wait_cluster(bar, parity);
  if (!ok) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
      if (mbar_try_wait_cluster(bar, parity)) {
        ok = true;
        break;
      }
      if (*abort_flag) break;
      if (globaltimer_ns() - t0 > prm.timeout_ns) {
        record_error(prm.p.err, kDevErrTimeout);
        *abort_flag = 1;
        break;
      }
    }
  }
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// bf16 split of 2n values into n packed words each: x1 truncated (fast, for
// the probabilities) or rounded to nearest (q, K, V), x2 = x - x1 rounded.
template <int N>
__device__ __forceinline__ void split_pack_trunc(const float* x, uint32_t* hi, uint32_t* lo) {
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float a = x[2 * i], b = x[2 * i + 1];
    hi[i] = pack_bf16_trunc(a, b);
    float ra, rb;
    fma2(ra, rb, bf16_trunc(a), bf16_trunc(b), -1.f, -1.f, a, b);  // x - x1, exact
    lo[i] = pack_bf16_rn(ra, rb);
  }
}
template <int N>
__device__ __forceinline__ void split_pack_rn(const float* x, uint32_t* hi, uint32_t* lo) {
#pragma unroll
  for (int i = 0; i < N; ++i) {
    float h0, h1;
    hi[i] = pack_bf16_rn_keep(x[2 * i], x[2 * i + 1], h0, h1);
    lo[i] = pack_bf16_rn(x[2 * i] - h0, x[2 * i + 1] - h1);
  }
}

template <bool kF32, int kSplit>
__global__ void __launch_bounds__(threads_of<kF32>(), 1)
tc_bf16_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
               const Params prm) {
  constexpr bool kTail = kSplit > 1;
  using L = Layout<kF32>;
  constexpr uint32_t kColO = col_o<kF32>();
  constexpr uint32_t kSmemK = L::kSmemK, kSmemV = L::kSmemV, kSmemBar = L::kSmemBar, kNumBars = L::kNumBars;
  constexpr uint32_t kSmemRed = L::kSmemRed, kSmemLsum = L::kSmemLsum, kStageBytes = L::kStageBytes;
  constexpr int kKS = L::kKS, kVS = L::kVS;
  constexpr uint32_t kColS = col_s<kF32>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const Bars bars = carve_bars<kF32>(smem);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kSmemBar + kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemBar + kNumBars * 8 + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKS; ++s) {
      mbar_init(&bars.kfull[s], 1);
      mbar_init(&bars.kconv[s], kConvWarpsPerOperand);
      mbar_init(&bars.kempty[s], 1);
    }
    for (int s = 0; s < kVS; ++s) {
      mbar_init(&bars.vconv[s], kConvWarpsPerOperand);
      mbar_init(&bars.vfull[s], 1);
      mbar_init(&bars.vempty[s], 1);
    }
    for (int b = 0; b < kNumS; ++b) {
      mbar_init(&bars.sfull[b], 1);
      mbar_init(&bars.pfull[b], kSoftmaxWarps);
      mbar_init(&bars.odone[b], 1);
    }
    mbar_init(bars.qready, kSoftmaxWarps);
    mbar_init(&bars.drain[0], 1);
    mbar_init(&bars.drain[1], 1);
    for (int q = 0; q < 4; ++q) mbar_init(&bars.pair[q], 2);
    if constexpr (kTail) {
      mbar_init(bars.partner, 1);
      mbar_init(bars.slotfree, kSoftmaxWarps * 32);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kQkWarp) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kKProducerWarp && lane == 0) tma_prefetch_desc(&tmk);
  if (warp == kVProducerWarp && lane == 0) tma_prefetch_desc(&tmv);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  if constexpr (kTail) {
    // Every CTA of the cluster is running and its barriers initialised before
    // any can touch another's shared memory.
    cluster_sync_all();
  } else {
    // A tail launch after this one (a programmatic dependent) may start its
    // blocks on SMs as soon as blocks of this grid leave them.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }
  const uint32_t rank = kTail ? cluster_ctarank() : 0u;

  const int cta = blockIdx.x, grid = gridDim.x;
  const Problem& p = prm.p;

  if (warp == kKProducerWarp || warp == kVProducerWarp) {
    // ------------------------------------------------------------ producers
    const bool is_k = warp == kKProducerWarp;
    if (lane == 0) {
      int n = 0;
      for (int k = 0;; ++k) {
        const int u = work_unit<kSplit>(k, cta, grid, prm);
        if (u >= prm.n_units) break;
        const Unit w = decode_unit(u, prm);
        int jb, je;
        unit_range<kSplit>(w, rank, &jb, &je);
        const int kStages = is_k ? kKS : kVS;
        for (int j = jb; j < je; ++j, ++n) {
          const int st = n % kStages;
          uint64_t* freed = is_k ? &bars.kempty[st] : &bars.vempty[st];
          if (n >= kStages && !wait_bar(freed, ((n / kStages) - 1) & 1, prm, abort_flag)) goto producer_done;
          uint64_t* full = is_k ? &bars.kfull[st] : &bars.vfull[st];
          uint8_t* dst = smem + (is_k ? kSmemK : kSmemV) + st * kStageBytes;
          mbar_arrive_expect_tx(full, kStageBytes);
          if (kF32) {  // d 0-31 and d 32-63 of the head, 128 rows each
            tma_load_2d(dst, is_k ? &tmk : &tmv, full, w.g * kD, j * kBc);
            tma_load_2d(dst + kOperandBytes, is_k ? &tmk : &tmv, full, w.g * kD + 32, j * kBc);
          } else {
            tma_load_2d(dst, is_k ? &tmk : &tmv, full, w.g * kD, j * kBc);
          }
        }
      }
    producer_done:
      if (*abort_flag) {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) __nanosleep(1000);
      }
    }
    __syncwarp();
  } else if (warp == kQkWarp || warp == kPvWarp) {
    // ---------------------------------------------------------- MMA issuers
    const bool is_qk = warp == kQkWarp;
    if (lane == 0) {
      int n = 0, lu = 0;
      for (int k = 0;; ++k) {
        const int u = work_unit<kSplit>(k, cta, grid, prm);
        if (u >= prm.n_units) break;
        const Unit w = decode_unit(u, prm);
        int jb, je;
        unit_range<kSplit>(w, rank, &jb, &je);
        if constexpr (kTail) {
          if (jb == je) continue;  // no tiles here (its Q is not loaded either)
        }
        if (is_qk) {
          if (!wait_bar(bars.qready, lu & 1, prm, abort_flag)) goto mma_done;
          tc_fence_after();
        }
        for (int j = jb; j < je; ++j, ++n) {
          const int b = n % kNumS;
          const int st = n % (is_qk ? kKS : kVS);
          const int kStages = is_qk ? kKS : kVS;
          if (is_qk) {
            // S buffer b is free once PV(n-3) has read P(n-3) from it; odone[b]
            // cannot be further ahead, since PV(n) needs S(n), issued below.
            if (!wait_bar(kF32 ? &bars.kconv[st] : &bars.kfull[st], (n / kStages) & 1, prm, abort_flag))
              goto mma_done;
            if (n >= kNumS && !wait_bar(&bars.odone[b], ((n / kNumS) - 1) & 1, prm, abort_flag)) goto mma_done;
            tc_fence_after();
            const uint32_t kb = smem_u32(smem + kSmemK + st * kStageBytes);
            const uint32_t d = tmem + kColS + b * 128;
            if (kF32) {  // q1 | q2 from shared memory
              const uint32_t qb = smem_u32(smem + L::kSmemQ);
#pragma unroll
              for (int s = 0; s < 4; ++s)
                mma_f16_ss(d, sdesc_sw128(qb + s * 32), sdesc_sw128(kb + s * 32), kIdescQK, s > 0);
#pragma unroll
              for (int s = 0; s < 4; ++s)
                mma_f16_ss(d, sdesc_sw128(qb + s * 32), sdesc_sw128(kb + kOperandBytes + s * 32), kIdescQK, 1);
#pragma unroll
              for (int s = 0; s < 4; ++s)
                mma_f16_ss(d, sdesc_sw128(qb + kOperandBytes + s * 32), sdesc_sw128(kb + s * 32), kIdescQK, 1);
            } else {
#pragma unroll
              for (int s = 0; s < 4; ++s)
                mma_f16_ts(d, tmem + kColQhi + s * 8, sdesc_sw128(kb + s * 32), kIdescQK, s > 0);
#pragma unroll
              for (int s = 0; s < 4; ++s)
                mma_f16_ts(d, tmem + kColQlo + s * 8, sdesc_sw128(kb + s * 32), kIdescQK, 1);
            }
            mma_commit(&bars.sfull[b]);
            mma_commit(&bars.kempty[st]);
          } else {
            if (!wait_bar(&bars.pfull[b], (n / kNumS) & 1, prm, abort_flag)) goto mma_done;
            if (!wait_bar(kF32 ? &bars.vconv[st] : &bars.vfull[st], (n / kStages) & 1, prm, abort_flag))
              goto mma_done;
            tc_fence_after();
            const uint32_t vb = smem_u32(smem + kSmemV + st * kStageBytes);
            const uint32_t phi = tmem + kColS + b * 128;
            const bool first = j == jb;
            if (kF32) {
#pragma unroll
              for (int s = 0; s < 8; ++s)  // [p1 v1 | p1 v2]: v2 is the N block kOperandBytes further
                mma_f16_ts(tmem + kColO, phi + s * 8, sdesc_sw128_mn(vb + s * 2048, kOperandBytes), kIdescPV128,
                           (first && s == 0) ? 0u : 1u);
            } else {
#pragma unroll
              for (int s = 0; s < 8; ++s)  // 16 keys per step: 2048 bytes of V rows
                mma_f16_ts(tmem + kColO, phi + s * 8, sdesc_sw128_mn(vb + s * 2048), kIdescPV,
                           (first && s == 0) ? 0u : 1u);
            }
#pragma unroll
            for (int s = 0; s < 8; ++s)
              mma_f16_ts(tmem + kColO, phi + 64 + s * 8, sdesc_sw128_mn(vb + s * 2048), kIdescPV, 1);
            mma_commit(&bars.odone[b]);
            mma_commit(&bars.vempty[st]);
          }
        }
        ++lu;
      }
    mma_done:
      if (*abort_flag) {
        uint64_t* drain = &bars.drain[is_qk ? 0 : 1];
        mma_commit(drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < prm.timeout_ns) {
        }
      }
    }
    __syncwarp();
  } else if (warp >= kFirstConvWarp) {
    // ---------------------------------------------- converters (fp32 cache)
    // Lane = one key. Its fp32 row lies in two 128-byte rows (d 0-31 in the
    // first region, d 32-63 in the second); x1 of the key goes to the same row
    // of the first region and x2 to the same row of the second, so each lane
    // rewrites exactly the bytes it read. 16-byte accesses of a quarter-warp hit
    // 8 consecutive rows at one logical chunk: 8 distinct bank groups under the
    // swizzle.
    if (kF32) {
      const bool is_k = warp < kFirstConvWarp + kConvWarpsPerOperand;
      const int cw = (warp - kFirstConvWarp) % kConvWarpsPerOperand;
      int n = 0;
      for (int k = 0;; ++k) {
        const int u = work_unit<kSplit>(k, cta, grid, prm);
        if (u >= prm.n_units) break;
        const Unit w = decode_unit(u, prm);
        int jb, je;
        unit_range<kSplit>(w, rank, &jb, &je);
        const int kStages = is_k ? kKS : kVS;
        for (int j = jb; j < je; ++j, ++n) {
          const int st = n % kStages;
          if (!wait_bar_warp(is_k ? &bars.kfull[st] : &bars.vfull[st], (n / kStages) & 1, prm, abort_flag))
            goto conv_done;
          uint8_t* base = smem + (is_k ? kSmemK : kSmemV) + st * kStageBytes;
#pragma unroll 1
          for (int r = 0; r < 2; ++r) {
            const uint32_t key = (uint32_t)(64 * cw + 32 * r + lane);
            float x[64];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int c4 = 0; c4 < 8; ++c4) {
                const float4 v = *reinterpret_cast<const float4*>(base + h * kOperandBytes +
                                                                  sw128(key * 128u + c4 * 16u));
                x[h * 32 + c4 * 4 + 0] = v.x;
                x[h * 32 + c4 * 4 + 1] = v.y;
                x[h * 32 + c4 * 4 + 2] = v.z;
                x[h * 32 + c4 * 4 + 3] = v.w;
              }
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
              uint32_t hi[4], lo[4];
              split_pack_rn<4>(x + c8 * 8, hi, lo);
              const uint32_t off = sw128(key * 128u + c8 * 16u);
              *reinterpret_cast<uint4*>(base + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
              *reinterpret_cast<uint4*>(base + kOperandBytes + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(is_k ? &bars.kconv[st] : &bars.vconv[st]);
        }
      }
    }
  conv_done:;
  } else {
    // -------------------------------------------------- softmax (warps 0-7)
    const int rq = warp & 3;         // TMEM lanes 32 rq .. + 31
    const int kh = warp >> 2;        // keys 64 kh .. + 63 of every tile; head dims 32 kh .. + 31
    const int row = rq * 32 + lane;
    const uint32_t lane_tmem = tmem + ((uint32_t)(rq * 32) << 16);
    float* red = reinterpret_cast<float*>(smem + kSmemRed);
    float* lred = reinterpret_cast<float*>(smem + kSmemLsum);
    const float c = kLog2e * kScale;
    const float stale = kStaleLog2 / c;
    int n = 0;

    uint32_t pc = 0;
    auto pair_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.pair[rq]);
      const bool ok = wait_bar_warp(&bars.pair[rq], pc & 1, prm, abort_flag);
      ++pc;
      return ok;
    };

    // This warp's 32 head dims of the row's query, split into bf16 hi/lo.
    auto load_q = [&](const Unit& w) {
      const int pos = w.t0 + (row >> 2);
      const float* src = p.q + ((size_t)pos * kHQ + w.g * kGroup + (row & 3)) * kD + kh * 32;
      float x[32];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (pos < p.C) v = __ldg(reinterpret_cast<const float4*>(src + i));
        x[i] = v.x;
        x[i + 1] = v.y;
        x[i + 2] = v.z;
        x[i + 3] = v.w;
      }
      uint32_t hi[16], lo[16];
      split_pack_rn<16>(x, hi, lo);
      if (kF32) {  // this warp's 32 dims: 16-byte chunks 4 kh .. 4 kh + 3 of the row's 128-byte swizzle row
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t off = sw128((uint32_t)row * 128u + (uint32_t)(kh * 4 + c) * 16u);
          *reinterpret_cast<uint4*>(smem + L::kSmemQ + off) = make_uint4(hi[4 * c], hi[4 * c + 1], hi[4 * c + 2], hi[4 * c + 3]);
          *reinterpret_cast<uint4*>(smem + L::kSmemQ + kOperandBytes + off) =
              make_uint4(lo[4 * c], lo[4 * c + 1], lo[4 * c + 2], lo[4 * c + 3]);
        }
        fence_proxy_async_smem();
      } else {
        tmem_st16(lane_tmem + kColQhi + kh * 16, hi);
        tmem_st16(lane_tmem + kColQlo + kh * 16, lo);
        tmem_wait_st();
        tc_fence_before();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.qready);
    };

    bool q_loaded = false;
    for (int k = 0;; ++k) {
      const int u = work_unit<kSplit>(k, cta, grid, prm);
      if (u >= prm.n_units) break;
      const Unit w = decode_unit(u, prm);
      int jb, je;
      unit_range<kSplit>(w, rank, &jb, &je);
      const bool has = jb < je;
      if (has && !q_loaded) load_q(w);
      q_loaded = false;
      float m_ref = -INFINITY, l = 0.f;
      const int pos = w.t0 + (row >> 2);
      const int limit = p.P + pos;
      for (int j = jb; j < je; ++j, ++n) {
        const int b = n % kNumS;
        const int j0 = j * kBc + kh * 64;
        const uint32_t sbuf = lane_tmem + kColS + b * 128;
        if (!wait_bar_warp(&bars.sfull[b], (n / kNumS) & 1, prm, abort_flag)) goto softmax_done;
        tc_fence_after();
        float s[64];
        tmem_ld32(sbuf + kh * 64, *reinterpret_cast<float(*)[32]>(&s[0]));
        tmem_ld32(sbuf + kh * 64 + 32, *reinterpret_cast<float(*)[32]>(&s[32]));
        tmem_wait_ld();
        if (j * kBc + kBc - 1 > p.P + w.t0) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (j0 + i > limit) s[i] = -INFINITY;
        }
        float mt = max3(s[0], s[1], s[2]);
#pragma unroll
        for (int i = 3; i < 63; i += 2) mt = max3(mt, s[i], s[i + 1]);
        mt = fmaxf(mt, s[63]);
        {
          // Both warps of the row set have read their S columns once they meet
          // here, so P may overwrite any of the buffer's columns afterwards.
          float* slot = red + (n & 1) * 256;
          slot[kh * 128 + row] = mt;
          if (!pair_sync()) goto softmax_done;
          mt = fmaxf(mt, slot[(kh ^ 1) * 128 + row]);
        }
        float alpha = 1.f;
        if (m_ref == -INFINITY || mt > m_ref + stale) {
          const float m_new = fmaxf(m_ref, mt);
          alpha = (m_ref == -INFINITY) ? 0.f : ex2((m_ref - m_new) * c);
          m_ref = m_new;
        }
        const float mc = m_ref == -INFINITY ? 0.f : m_ref * c;
        float l0 = 0.f, l1 = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float* x = s + half * 32 + i;
            fma2(x[0], x[1], x[0], x[1], c, c, -mc, -mc);
            x[0] = ex2(x[0]);
            x[1] = ex2(x[1]);
            add2(l0, l1, l0, l1, x[0], x[1]);
          }
          uint32_t hi[16], lo[16];
          split_pack_trunc<16>(s + half * 32, hi, lo);
          tmem_st16(sbuf + kh * 32 + half * 16, hi);
          tmem_st16(sbuf + 64 + kh * 32 + half * 16, lo);
        }
        l = fmaf(l, alpha, l0 + l1);
        tmem_wait_st();
        // O is rescaled only when the reference maximum moved, after PV(n-1)
        // completes (odone[(n-1) % 3] cannot be a phase further: PV(n+2) needs
        // P(n+2) from these warps).
        if (j > jb && __any_sync(0xffffffffu, alpha != 1.f)) {
          const int pb = (n - 1) % kNumS;
          if (!wait_bar_warp(&bars.odone[pb], ((n - 1) / kNumS) & 1, prm, abort_flag)) goto softmax_done;
          tc_fence_after();
          float o[32];
          tmem_ld32(lane_tmem + kColO + kh * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(lane_tmem + kColO + kh * 32, o);
          if (kF32) {
            tmem_ld32(lane_tmem + kColO + 64 + kh * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(lane_tmem + kColO + 64 + kh * 32, o);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.pfull[b]);
      }
      {
        const int u_next = work_unit<kSplit>(k + 1, cta, grid, prm);
        if (u_next < prm.n_units) {
          load_q(decode_unit(u_next, prm));
          q_loaded = true;
        }
      }
      lred[kh * 128 + row] = l;
      if (!pair_sync()) goto softmax_done;
      l += lred[(kh ^ 1) * 128 + row];
      if constexpr (kSplit == 3 || kSplit == 4 || kSplit == 8 || kSplit == 12) {
        // A unit split over a cluster of three, four, eight or twelve, as over
        // a pair below.
        // Senders stage their shares in their own K rings; a receiver, once
        // its last PV has completed (its K and V rings are then idle), takes
        // up to three shares in consecutive slots there and folds them into
        // its own partial, m = the largest maximum of a part with tiles, each
        // part weighted by e^(m_s - m). Four: ranks 1-3 send to rank 0. Eight:
        // ranks 2-4 send to rank 0 and ranks 5-7 to rank 1; rank 1 then sends
        // its merged partial to rank 0's slot 0, once rank 0 has folded in
        // its first three. Three: ranks 1-2 send to rank 0. Twelve: ranks 4-11
        // send to ranks 0-3, two each; rank 0 folds in its two, then takes
        // ranks 1-3's merged partials.
        static_assert(kSmemK + 3 * kShareBytes <= kSmemBar, "three shares fit in the K and V rings");
        float o[32];
        if (has) {
          const int pb = (n - 1) % kNumS;
          if (!wait_bar_warp(&bars.odone[pb], ((n - 1) / kNumS) & 1, prm, abort_flag)) goto softmax_done;
          tc_fence_after();
          tmem_ld32(lane_tmem + kColO + kh * 32, o);
          tmem_wait_ld();
          if (kF32) {
            float o2[32];
            tmem_ld32(lane_tmem + kColO + 64 + kh * 32, o2);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] += o2[i];
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0.f;
        }
        uint8_t* share = smem + kSmemK;
        auto share_offset = [&](int i) -> uint32_t {  // this thread's chunk i (4 floats) of its row half
          return (uint32_t)kh * 16384u + (uint32_t)row * 128u + (uint32_t)((i ^ (row & 7)) * 16);
        };
        auto receive = [&](uint32_t first, int nslots, uint32_t phase) -> bool {
          for (int r = 0; r < nslots; ++r)
            mbar_arrive_remote(mapa_shared(smem_u32(bars.slotfree), first + (uint32_t)r));
          if (row == 0 && kh == 0) mbar_arrive_expect_tx(bars.partner, (uint32_t)nslots * kShareBytes);
          if (!wait_bar_cluster_warp(bars.partner, phase, prm, abort_flag)) return false;
          float m = l > 0.f ? m_ref : -INFINITY;
#pragma unroll 3
          for (int r = 0; r < nslots; ++r) {
            const float* ml = reinterpret_cast<const float*>(share + r * kShareBytes + kShareO);
            if (ml[128 + row] > 0.f) m = fmaxf(m, ml[row]);
          }
          const float e0 = l > 0.f ? ex2((m_ref - m) * c) : 0.f;
          float den = e0 * l;
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= e0;
#pragma unroll 3
          for (int r = 0; r < nslots; ++r) {
            const uint8_t* slot = share + r * kShareBytes;
            const float* ml = reinterpret_cast<const float*>(slot + kShareO);
            const float lr = ml[128 + row];
            const float er = lr > 0.f ? ex2((ml[row] - m) * c) : 0.f;
            den = fmaf(er, lr, den);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 x = *reinterpret_cast<const float4*>(slot + share_offset(i));
              o[4 * i] = fmaf(er, x.x, o[4 * i]);
              o[4 * i + 1] = fmaf(er, x.y, o[4 * i + 1]);
              o[4 * i + 2] = fmaf(er, x.z, o[4 * i + 2]);
              o[4 * i + 3] = fmaf(er, x.w, o[4 * i + 3]);
            }
          }
          m_ref = m;
          l = den;
          return true;
        };
        // Stage (o, m_ref, l) in slot 0 of this CTA (each thread its own row
        // half, so a receiver overwrites only what it has read) and copy it
        // in bulk into slot `slot` of CTA `to` once that CTA's slots are free.
        auto send = [&](uint32_t to, uint32_t slot) -> bool {
          // After a receive, both warps of the row set must have read slot 0's
          // maxima and sums before the kh = 0 warp overwrites them.
          if (((kSplit == 8 && rank == 1) || (kSplit == 12 && rank >= 1 && rank <= 3)) && !pair_sync()) return false;
          float* ml = reinterpret_cast<float*>(share + kShareO);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4*>(share + share_offset(i)) =
                make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
          if (kh == 0) {
            ml[row] = m_ref;
            ml[128 + row] = l;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (!wait_bar_cluster_warp(bars.slotfree, 0, prm, abort_flag)) return false;
          if ((row & 31) == 0) {
            const uint32_t bar = mapa_shared(smem_u32(bars.partner), to);
            const uint32_t dst_slot = smem_u32(share) + slot * kShareBytes;  // the same offset in `to`
            const uint32_t part = (uint32_t)kh * 16384u + (uint32_t)row * 128u;
            bulk_copy_to_cluster(mapa_shared(dst_slot + part, to), share + part, 32 * 128, bar);
            if (kh == 0) {
              bulk_copy_to_cluster(mapa_shared(dst_slot + kShareO + row * 4, to), ml + row, 32 * 4, bar);
              bulk_copy_to_cluster(mapa_shared(dst_slot + kShareO + (128 + row) * 4, to), ml + 128 + row, 32 * 4,
                                   bar);
            }
          }
          return true;
        };
        bool ok;
        if (rank == 0) {
          ok = kSplit == 12  ? (receive(4, 2, 0) && receive(1, 3, 1))
               : kSplit == 8 ? (receive(2, 3, 0) && receive(1, 1, 1))
                             : receive(1, kSplit - 1, 0);
          if (ok && pos < p.C) {
            const float inv = 1.f / l;  // > 0: the unit sees at least key 0
            float* dst = p.out + ((size_t)pos * kHQ + w.g * kGroup + (row & 3)) * kD + kh * 32;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              *reinterpret_cast<float4*>(dst + 4 * i) =
                  make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
          }
        } else if (kSplit == 12) {
          ok = rank <= 3 ? (receive(2 * rank + 4, 2, 0) && send(0, rank - 1))
                         : send((rank - 4) >> 1, (rank - 4) & 1);
        } else if (kSplit != 8) {
          ok = send(0, rank - 1);
        } else if (rank == 1) {
          ok = receive(5, 3, 0) && send(0, 0);
        } else {
          ok = rank < 5 ? send(0, rank - 2) : send(1, rank - 5);
        }
        if (!ok) goto softmax_done;
        tc_fence_before();
        continue;
      }
      if constexpr (kSplit == 2) {
        // A unit split over the CTA pair; this thread holds 32 of its row's 64
        // output dims (head dims 32 kh ..), and l and the reference maximum of
        // this CTA's key tiles (none when it got no tile). The output is only
        // written: rank 1 stages its unnormalised O, m and l in its own K ring;
        // rank 0, once its last PV has completed (its K ring is then idle),
        // tells rank 1 so, and each warp of rank 1 copies its part in bulk
        // (cp.async.bulk between the CTAs' shared memories) into rank 0's K
        // ring, the bytes completing on rank 0's partner barrier; rank 0
        // merges, m = max(m0, m1) with weights e^(m_s - m) (in log2 units,
        // (m_s - m) c), one reciprocal per row, and stores.
        float o[32];
        if (has) {
          const int pb = (n - 1) % kNumS;
          if (!wait_bar_warp(&bars.odone[pb], ((n - 1) / kNumS) & 1, prm, abort_flag)) goto softmax_done;
          tc_fence_after();
          tmem_ld32(lane_tmem + kColO + kh * 32, o);
          tmem_wait_ld();
          if (kF32) {
            float o2[32];
            tmem_ld32(lane_tmem + kColO + 64 + kh * 32, o2);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] += o2[i];
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = 0.f;
        }
        // The share: [head-dim half kh][row][32 floats], a row's 16-byte chunk
        // i at chunk i ^ (row mod 8), then the 128 maxima and the 128 sums.
        uint8_t* share = smem + kSmemK;
        float* ml = reinterpret_cast<float*>(share + kShareO);
        auto share_offset = [&](int i) -> uint32_t {  // this thread's chunk i (4 floats) of its row half
          return (uint32_t)kh * 16384u + (uint32_t)row * 128u + (uint32_t)((i ^ (row & 7)) * 16);
        };
        const uint32_t peer = rank ^ 1u;
        if (rank == 1) {
          // Stage in this CTA's own K ring (its MMAs are complete); once rank
          // 0's K ring is free, each warp copies its 32 row halves (and, for
          // kh = 0, their maxima and sums) in bulk into rank 0's, completing
          // on rank 0's partner barrier.
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<float4*>(share + share_offset(i)) =
                make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
          if (kh == 0) {
            ml[row] = m_ref;
            ml[128 + row] = l;
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (!wait_bar_cluster_warp(bars.slotfree, 0, prm, abort_flag)) goto softmax_done;
          if ((row & 31) == 0) {
            const uint32_t bar = mapa_shared(smem_u32(bars.partner), peer);
            uint8_t* part = share + (uint32_t)kh * 16384u + (uint32_t)row * 128u;
            bulk_copy_to_cluster(mapa_shared(smem_u32(part), peer), part, 32 * 128, bar);
            if (kh == 0) {
              bulk_copy_to_cluster(mapa_shared(smem_u32(ml + row), peer), ml + row, 32 * 4, bar);
              bulk_copy_to_cluster(mapa_shared(smem_u32(ml + 128 + row), peer), ml + 128 + row, 32 * 4, bar);
            }
          }
        } else {
          mbar_arrive_remote(mapa_shared(smem_u32(bars.slotfree), peer));
          if (row == 0 && kh == 0) mbar_arrive_expect_tx(bars.partner, kShareBytes);
          if (!wait_bar_cluster_warp(bars.partner, 0, prm, abort_flag)) goto softmax_done;
          const float m1 = ml[row], l1 = ml[128 + row];
          const float m = fmaxf(l > 0.f ? m_ref : -INFINITY, l1 > 0.f ? m1 : -INFINITY);
          const float e0 = l > 0.f ? ex2((m_ref - m) * c) : 0.f;
          const float e1 = l1 > 0.f ? ex2((m1 - m) * c) : 0.f;
          const float inv = 1.f / fmaf(e0, l, e1 * l1);  // > 0: the unit sees at least key 0
          if (pos < p.C) {
            float* dst = p.out + ((size_t)pos * kHQ + w.g * kGroup + (row & 3)) * kD + kh * 32;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 x1 = *reinterpret_cast<const float4*>(share + share_offset(i));
              *reinterpret_cast<float4*>(dst + 4 * i) =
                  make_float4(fmaf(e0, o[4 * i], e1 * x1.x) * inv, fmaf(e0, o[4 * i + 1], e1 * x1.y) * inv,
                              fmaf(e0, o[4 * i + 2], e1 * x1.z) * inv, fmaf(e0, o[4 * i + 3], e1 * x1.w) * inv);
            }
          }
        }
        tc_fence_before();
        continue;
      }
      {
        const int pb = (n - 1) % kNumS;
        if (!wait_bar_warp(&bars.odone[pb], ((n - 1) / kNumS) & 1, prm, abort_flag)) goto softmax_done;
      }
      tc_fence_after();
      {
        float a[32];
        tmem_ld32(lane_tmem + kColO + kh * 32, a);
        tmem_wait_ld();
        if (kF32) {
          float a2[32];
          tmem_ld32(lane_tmem + kColO + 64 + kh * 32, a2);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) a[i] += a2[i];
        }
        if (pos < p.C) {
          float* dst = p.out + ((size_t)pos * kHQ + w.g * kGroup + (row & 3)) * kD + kh * 32;
          const float inv = 1.f / l;
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + i) = make_float4(a[i] * inv, a[i + 1] * inv, a[i + 2] * inv,
                                                              a[i + 3] * inv);
        }
      }
      tc_fence_before();
    }
  softmax_done:;
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if constexpr (kTail) {
    // No CTA of the cluster leaves while another may still write its shared
    // memory or arrive on its barriers.
    cluster_sync_all();
  }
  if (warp == kQkWarp) tmem_dealloc(tmem, kTmemCols);
  if constexpr (kTail) {
    // This grid ends only after the grid of whole units it overlaps: work
    // ordered after it on the stream sees both complete.
    asm volatile("griddepcontrol.wait;" ::: "memory");
  }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

// The driver's tensor-map encoder, looked up once (a function-local static is
// initialised once even when the first calls come from several threads).
PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      ptr = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

// k or v [rows][8][64] as a 2-D tensor (head * 64 + d, row); a box is 128
// bytes of one head's values (64 bf16, or 32 fp32: one swizzle row) x 128 rows.
int encode_kv_tile_map(const void* base, int rows, bool f32, CUtensorMap* map) {
  auto enc = encoder();
  if (!enc) return ATTN_ETMA;
  const cuuint32_t ones[2] = {1, 1};
  const cuuint64_t dims[2] = {(cuuint64_t)kHKV * kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kHKV * kD * (f32 ? 4 : 2)};
  const cuuint32_t box[2] = {(cuuint32_t)(f32 ? 32 : 64), (cuuint32_t)kBc};
  if (enc(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base),
          dims, strides, box, ones, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return ATTN_ETMA;
  return ATTN_OK;
}

struct DevState {
  bool ready[2] = {false, false};  // per cache type, its instantiations set up
  int num_sms = 0;
  int quads[2] = {0, 0};   // per cache type: clusters of four tail CTAs the device holds at once
  int octets[2] = {0, 0};  // and of eight
  int trios[2] = {0, 0};   // and of three
  int twelves[2] = {0, 0};  // and of twelve
};
DevState g_state[64];
std::mutex g_state_mu;

template <bool kF32>
int launch_impl(const Problem& p, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ECUDA;
  int num_sms = 0, quads = 0, octets = 0, trios = 0, twelves = 0;
  {
    std::lock_guard<std::mutex> lock(g_state_mu);
    DevState& st = g_state[dev];
    if (!st.ready[kF32]) {
      if (cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ATTN_ECUDA;
      if (cudaFuncSetAttribute(tc_bf16_kernel<kF32, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)Layout<kF32>::kSmemAlloc) != cudaSuccess ||
          cudaFuncSetAttribute(tc_bf16_kernel<kF32, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)Layout<kF32>::kSmemAlloc) != cudaSuccess ||
          cudaFuncSetAttribute(tc_bf16_kernel<kF32, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)Layout<kF32>::kSmemAlloc) != cudaSuccess ||
          cudaFuncSetAttribute(tc_bf16_kernel<kF32, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)Layout<kF32>::kSmemAlloc) != cudaSuccess ||
          cudaFuncSetAttribute(tc_bf16_kernel<kF32, 3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)Layout<kF32>::kSmemAlloc) != cudaSuccess ||
          cudaFuncSetAttribute(tc_bf16_kernel<kF32, 12>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)Layout<kF32>::kSmemAlloc) != cudaSuccess)
        return ATTN_ECUDA;
      // Clusters of twelve are a non-portable size: allowed per kernel (on
      // a device that refuses, no twelve-way split).
      const bool twelve_ok = cudaFuncSetAttribute(tc_bf16_kernel<kF32, 12>,
                                                  cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
      if (!twelve_ok) (void)cudaGetLastError();
      // How many clusters of three, four and eight fit at once (0 when a
      // query fails: no such split then).
      auto clusters_of = [&](int size, void (*kernel)(CUtensorMap, CUtensorMap, Params)) {
        cudaLaunchConfig_t qc = {};
        qc.gridDim = dim3(size * kHKV);
        qc.blockDim = dim3(threads_of<kF32>());
        qc.dynamicSmemBytes = Layout<kF32>::kSmemAlloc;
        cudaLaunchAttribute qa[1];
        qa[0].id = cudaLaunchAttributeClusterDimension;
        qa[0].val.clusterDim.x = size;
        qa[0].val.clusterDim.y = 1;
        qa[0].val.clusterDim.z = 1;
        qc.attrs = qa;
        qc.numAttrs = 1;
        int nc = 0;
        if (cudaOccupancyMaxActiveClusters(&nc, kernel, &qc) != cudaSuccess) {
          (void)cudaGetLastError();
          nc = 0;
        }
        return nc;
      };
      st.quads[kF32] = clusters_of(4, tc_bf16_kernel<kF32, 4>);
      st.octets[kF32] = clusters_of(8, tc_bf16_kernel<kF32, 8>);
      st.trios[kF32] = clusters_of(3, tc_bf16_kernel<kF32, 3>);
      st.twelves[kF32] = twelve_ok ? clusters_of(12, tc_bf16_kernel<kF32, 12>) : 0;
      st.ready[kF32] = true;
    }
    num_sms = st.num_sms;
    quads = st.quads[kF32];
    octets = st.octets[kF32];
    trios = st.trios[kF32];
    twelves = st.twelves[kF32];
  }
  alignas(64) CUtensorMap mk, mv;
  int rc = encode_kv_tile_map(p.k, p.P + p.C, kF32, &mk);
  if (rc == ATTN_OK) rc = encode_kv_tile_map(p.v, p.P + p.C, kF32, &mv);
  if (rc != ATTN_OK) return rc;
  Params prm;
  prm.p = p;
  prm.n_qtiles = (p.C + kBq - 1) / kBq;
  prm.n_units = prm.n_qtiles * kHKV;
  prm.timeout_ns = 2000000000ull;
  prm.unit_base = 0;
  const int grid = prm.n_units < num_sms ? prm.n_units : num_sms;
  // Split units, as for the split-TF32 kernel: with several rounds, a short
  // last round's units go to a second grid of CTA pairs that each split one;
  // with at most half as many units as SMs, every unit is split over a pair.
  // Rules as there (the last round: units of 1024 keys or more; every unit:
  // the longest of 1024 or more, these 128-key tiles making shorter halves
  // too small). With the bulk-copy hand-off the last-round split measured
  // 329.7 -> 334.1 TFLOP/s at the serving chunk for bf16x3 (the bf16 cache
  // unchanged), and splitting every unit of small chunks against 1024-8192
  // keys 1.1-1.6x (with the remote stores both had been kept to units of
  // 8192 keys or more). Every unit is split over a cluster of four instead
  // when the device holds one for every unit (chunks of 128 rows or less on
  // 152 SMs: measured 1.3-1.8x faster than pairs against 4096-32768 keys,
  // 1.1x against 1200-2500), and over eight when it holds a cluster of eight
  // for every unit and the longest unit sees 2048 keys or more (chunks of 32
  // rows or less: 1.6-1.7x faster than fours against 32768 keys; over twelve,
  // a non-portable size, from 8192 keys), and over
  // three when it holds a cluster of three for every unit (chunks of 129-184
  // rows: 1.4x faster than pairs against 32768 keys).
  Params main_prm = prm, tail_prm = prm;
  int main_grid = grid, tail_units = 0, split = 2;
  if (prm.n_units > grid) {
    const int full = prm.n_units / grid * grid;
    const int rem = prm.n_units - full;
    if (rem > 0 && 2 * rem <= (num_sms & ~1) && unit_keys(p.P, p.C, 0, kBq) >= 1024) {
      main_prm.n_units = full;
      tail_prm.unit_base = full;
      tail_units = rem;
      // These units too go to the largest clusters the device holds one of for
      // every such unit (measured against pairs, 16 or 24 units over fours:
      // 1.03-1.19x for chunks of 660-1900 rows against 2048-30000 keys).
      if (rem <= twelves && unit_keys(p.P, p.C, 0, kBq) >= 8192)
        split = 12;
      else if (rem <= octets && unit_keys(p.P, p.C, 0, kBq) >= 2048)
        split = 8;
      else if (rem <= quads)
        split = 4;
      else if (rem <= trios)
        split = 3;
    } else if (rem > num_sms / 2 && rem <= 2 * trios && unit_keys(p.P, p.C, 0, kBq) >= 8192) {
      // A last round of more than half as many units as SMs: over clusters of
      // three in two waves, when its units are long (measured 1.03-1.14x for
      // chunks of 928-1568 rows against 8192-30000 keys; 0.91-1.03x against
      // 2048-4096).
      main_prm.n_units = full;
      tail_prm.unit_base = full;
      tail_units = rem;
      split = 3;
    }
  } else if (2 * prm.n_units <= num_sms && unit_keys(p.P, p.C, (prm.n_qtiles - 1) * kBq, kBq) >= 1024) {
    // Measured: splitting only some of the units (more than half as many
    // units as SMs) costs more than it gains.
    main_prm.n_units = 0;
    tail_prm.unit_base = 0;
    tail_units = prm.n_units;
    if (prm.n_units <= twelves && unit_keys(p.P, p.C, (prm.n_qtiles - 1) * kBq, kBq) >= 8192)
      split = 12;
    else if (prm.n_units <= octets && unit_keys(p.P, p.C, (prm.n_qtiles - 1) * kBq, kBq) >= 2048)
      split = 8;
    else if (prm.n_units <= 2 * twelves && unit_keys(p.P, p.C, (prm.n_qtiles - 1) * kBq, kBq) >= 16384)
      split = 12;  // more units than clusters of eight: twelves in two waves (long units only)
    else if (prm.n_units <= quads)
      split = 4;
    else if (prm.n_units <= trios)
      split = 3;
  } else if (prm.n_units <= 2 * trios && unit_keys(p.P, p.C, (prm.n_qtiles - 1) * kBq, kBq) >= 8192) {
    // A partial round of more than half as many units as SMs: every unit over
    // a cluster of three, the clusters running in two waves as the device
    // frees SMs (measured 1.15-1.38x for chunks of 320-352 rows against
    // 8192-32768 keys; below that many keys, or with more units, whole units
    // stay faster).
    main_prm.n_units = 0;
    tail_prm.unit_base = 0;
    tail_units = prm.n_units;
    split = 3;
  }
  if (main_prm.n_units > 0) {
    tc_bf16_kernel<kF32, 1><<<main_grid, threads_of<kF32>(), Layout<kF32>::kSmemAlloc, stream>>>(mk, mv,
                                                                                                   main_prm);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ELAUNCH;
  }
  if (tail_units == 0) return ATTN_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(split * tail_units);
  cfg.blockDim = dim3(threads_of<kF32>());
  cfg.dynamicSmemBytes = Layout<kF32>::kSmemAlloc;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = split;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = main_prm.n_units > 0 ? 2 : 1;  // a dependent only of a whole-unit grid
  auto* tail = split == 8   ? tc_bf16_kernel<kF32, 8>
               : split == 4 ? tc_bf16_kernel<kF32, 4>
               : split == 3 ? tc_bf16_kernel<kF32, 3>
               : split == 12 ? tc_bf16_kernel<kF32, 12>
                            : tc_bf16_kernel<kF32, 2>;
  if (cudaLaunchKernelEx(&cfg, tail, mk, mv, tail_prm) != cudaSuccess) return ATTN_ELAUNCH;
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ELAUNCH;
}

}  // namespace

int launch_tc_bf16(const Problem& p, cudaStream_t stream) { return launch_impl<false>(p, stream); }

int launch_tc_bf16x3(const Problem& p, cudaStream_t stream) { return launch_impl<true>(p, stream); }

}  // namespace attn
