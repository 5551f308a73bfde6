// tc.cu -- the main path: persistent, warp-specialised flash prefill on the
// sm_103a tensor cores (tcgen05, TMEM accumulators, TMA staging).
//
// What it computes is the tiled online-softmax attention of "Inference
// Attention 2: Flash Prefill Against a Cached Prefix" (Lesson): a chunk of C
// rows at positions P..P+C-1 against keys 0..P+C-1, row i seeing j <= P+i,
// query head h reading KV head h/4, scale 1/8. Per tile with maximum m_tile:
// m_new = max(m_old, m_tile), alpha = exp(m_old - m_new), l and the
// accumulator rescaled by alpha, one division by l at the very end.
//
// Work unit: 32 chunk positions x the 4 query heads that share KV head g
// (GQA packing, "FlashAttention and inference kernels", GQA read
// amplification) = 128 rows, one row per TMEM lane, row r = 4 (pos - t0) +
// (head - 4 g). Keys are visited in tiles of 64; tiles beyond the unit's last
// visible key are never loaded and only tiles that cross the diagonal are
// masked (same page, "How FlashAttention evolved", the causal mask).
//
// Contractions: fp32 split-TF32. Every operand x is split into hi = x with the
// 13 low mantissa bits cleared (exactly tf32) and lo = x - hi (exact in fp32);
// a product is accumulated as hi*hi + hi*lo + lo*hi on the tensor cores in
// fp32, dropping only lo*lo (relative size 2^-20). QK^T: A = Q (hi and lo in
// TMEM), B = K (shared memory, K-major, 128-byte swizzle). PV: A = P (hi and lo
// in TMEM, P hi overwriting the S columns it came from), B = V^T (shared
// memory, written transposed by the converter warps).
//
// Warp roles (10 warps):
//   0-3  softmax: own TMEM lanes 0-127 (one row each); split Q into TMEM at the
//        start of a unit; per tile read S, mask, online softmax, write P hi/lo,
//        rescale O when the reference maximum moves; epilogue O / l -> out.
//   4    producer: TMA loads of Q, K and V tiles into the shared-memory rings.
//   5    MMA: allocates TMEM; one lane issues every tcgen05.mma and commit.
//   6-9  converters: K -> K lo; V -> V^T hi and V^T lo.
// Every wait is bounded; on expiry the kernel records ATTN_ETIMEOUT in the
// device error word, all roles wind down, and TMEM is freed.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace attn {
namespace {

using namespace tc;

constexpr int kBq = 32;         // chunk positions per unit
constexpr int kM = kBq * kGroup;  // 128 rows = TMEM lanes
constexpr int kBc = 64;         // keys per tile
constexpr int kKStages = 3;     // K ring (raw K as tf32 hi after the in-place split, plus K lo)
constexpr int kVRawStages = 2;  // raw V landing ring
constexpr int kVStages = 2;     // V^T hi/lo ring

constexpr int kSoftmaxWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kFirstConvWarp = 6;
constexpr int kConvWarps = 4;
constexpr int kThreads = 32 * (kFirstConvWarp + kConvWarps);

// TMEM columns (fp32, one per column).
constexpr uint32_t kColQhi = 0;
constexpr uint32_t kColQlo = 64;
constexpr uint32_t kColS = 128;    // two S buffers of 64 columns; P hi overwrites S
constexpr uint32_t kColPlo = 256;  // two P lo buffers of 64 columns
constexpr uint32_t kColO = 384;
constexpr uint32_t kTmemCols = 512;

// Shared memory (byte offsets from a 1024-aligned base). Every operand tile
// is a set of 128-byte-swizzled regions: rows of 128 bytes (32 floats).
constexpr uint32_t kQBytes = kM * kD * 4;                 // 32 KB: 2 d-half regions of 128 rows
constexpr uint32_t kKTileBytes = kBc * kD * 4;            // 16 KB: 2 d-half regions of 64 rows
constexpr uint32_t kSmemQ = 0;
constexpr uint32_t kSmemK = kSmemQ + kQBytes;                             // [stage][K | K lo]
constexpr uint32_t kSmemVRaw = kSmemK + kKStages * 2 * kKTileBytes;       // [stage][V]
constexpr uint32_t kSmemVT = kSmemVRaw + kVRawStages * kKTileBytes;       // [stage][V^T hi | V^T lo]
constexpr uint32_t kSmemBar = kSmemVT + kVStages * 2 * kKTileBytes;
constexpr uint32_t kNumBars = 3 * kKStages + 2 * kVRawStages + 2 * kVStages + 2 + 2 + 5;
constexpr uint32_t kSmemTotal = kSmemBar + kNumBars * 8 + 16;
constexpr uint32_t kSmemAlloc = kSmemTotal + 1024;  // slack to align the base

static_assert(kSmemAlloc <= 232448, "exceeds the 227 KB per-block shared memory limit");
static_assert(kM == 128 && kD == 64 && kBc == 64, "the MMA shapes below assume 128 x 64 x 64");

constexpr uint32_t kIdesc = idesc_tf32(128, 64);
// Keep a stale reference maximum while the new maximum exceeds it by at most
// this much in log2 units (p stays <= 2^8): l and O share the reference, so
// O / l is exact either way, and O needs no rescale.
constexpr float kStaleLog2 = 8.0f;
// The tensor core reads an fp32 operand as tf32 by ignoring its 13 low
// mantissa bits (measured on GB300 for both shared-memory and TMEM operands:
// 1 + 3 * 2^-12 reads as 1), so raw K already is tf32_hi(K) to the MMA and
// only K lo has to be written. Set to false to truncate K in place as well.
constexpr bool kHwTruncatesTf32 = true;

struct Params {
  Problem p;
  int n_units;
  int n_qtiles;
  unsigned long long timeout_ns;
  int fault_skip_first_k;  // test hook: never load the first K tile
};

struct Bars {
  uint64_t* kfull;   // [kKStages] TMA K landed
  uint64_t* kconv;   // [kKStages] K lo written (converter warps)
  uint64_t* kempty;  // [kKStages] QK done with the stage (MMA commit)
  uint64_t* vfull;   // [kVRawStages] TMA V landed
  uint64_t* vrfree;  // [kVRawStages] converters done reading raw V
  uint64_t* vconv;   // [kVStages] V^T hi/lo written
  uint64_t* vempty;  // [kVStages] PV done with the stage (MMA commit)
  uint64_t* sfull;   // [2] S buffer written (MMA commit)
  uint64_t* pfull;   // [2] P hi/lo written and O rescaled (softmax warps)
  uint64_t* odone;   // PV done (MMA commit)
  uint64_t* qfull;   // TMA Q landed
  uint64_t* qfree;   // softmax warps done reading the Q staging buffer
  uint64_t* qready;  // Q hi/lo in TMEM
  uint64_t* drain;   // MMA drain on abort
};

__device__ __forceinline__ Bars carve_bars(uint8_t* base) {
  uint64_t* b = reinterpret_cast<uint64_t*>(base + kSmemBar);
  Bars r;
  r.kfull = b; b += kKStages;
  r.kconv = b; b += kKStages;
  r.kempty = b; b += kKStages;
  r.vfull = b; b += kVRawStages;
  r.vrfree = b; b += kVRawStages;
  r.vconv = b; b += kVStages;
  r.vempty = b; b += kVStages;
  r.sfull = b; b += 2;
  r.pfull = b; b += 2;
  r.odone = b++;
  r.qfull = b++;
  r.qfree = b++;
  r.qready = b++;
  r.drain = b++;
  return r;
}

// The CTA's k-th unit in a snake order over units sorted longest first.
__device__ __forceinline__ int unit_index(int k, int cta, int grid) {
  return k * grid + ((k & 1) ? (grid - 1 - cta) : cta);
}

struct Unit {
  int t0, g, ntiles;
};
__device__ __forceinline__ Unit decode_unit(int u, const Params& prm) {
  Unit w;
  const int qt = prm.n_qtiles - 1 - u / kHKV;  // last q-tiles see the most keys
  w.g = u % kHKV;
  w.t0 = qt * kBq;
  const int nkeys = unit_keys(prm.p.P, prm.p.C, w.t0, kBq);
  w.ntiles = (nkeys + kBc - 1) / kBc;
  return w;
}

// Bounded wait that also gives up when another role has aborted.
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

// Every lane of the warp waits; the outcome is made warp-uniform so that the
// .sync.aligned tensor-memory instructions after it never run on a partial warp.
__device__ __forceinline__ bool wait_bar_warp(uint64_t* bar, uint32_t parity, const Params& prm,
                                              volatile int* abort_flag) {
  const bool ok = wait_bar(bar, parity, prm, abort_flag);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(kThreads, 1)
tc_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
          const __grid_constant__ CUtensorMap tmv, const Params prm) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const Bars bars = carve_bars(smem);
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kSmemBar + kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kSmemBar + kNumBars * 8 + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&bars.kfull[s], 1);
      mbar_init(&bars.kconv[s], kConvWarps);
      mbar_init(&bars.kempty[s], 1);
    }
    for (int s = 0; s < kVRawStages; ++s) {
      mbar_init(&bars.vfull[s], 1);
      mbar_init(&bars.vrfree[s], kConvWarps);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&bars.vconv[s], kConvWarps);
      mbar_init(&bars.vempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars.sfull[b], 1);
      mbar_init(&bars.pfull[b], kSoftmaxWarps);
    }
    mbar_init(bars.odone, 1);
    mbar_init(bars.qfull, 1);
    mbar_init(bars.qfree, kSoftmaxWarps);
    mbar_init(bars.qready, kSoftmaxWarps);
    mbar_init(bars.drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmq);
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const int cta = blockIdx.x, grid = gridDim.x;
  const Problem& p = prm.p;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      int n = 0, lu = 0;
      for (int k = 0;; ++k) {
        const int u = unit_index(k, cta, grid);
        if (u >= prm.n_units) break;
        const Unit w = decode_unit(u, prm);
        if (lu > 0 && !wait_bar(bars.qfree, (lu - 1) & 1, prm, abort_flag)) goto producer_done;
        mbar_arrive_expect_tx(bars.qfull, kQBytes);
        tma_load_3d(smem + kSmemQ, &tmq, bars.qfull, 0, w.g * kGroup, w.t0);
        tma_load_3d(smem + kSmemQ + kQBytes / 2, &tmq, bars.qfull, 32, w.g * kGroup, w.t0);
        for (int j = 0; j < w.ntiles; ++j, ++n) {
          const int j0 = j * kBc;
          const int ks = n % kKStages;
          if (n >= kKStages && !wait_bar(&bars.kempty[ks], ((n / kKStages) - 1) & 1, prm, abort_flag))
            goto producer_done;
          uint8_t* kdst = smem + kSmemK + ks * 2 * kKTileBytes;
          if (!(prm.fault_skip_first_k && n == 0)) {
            mbar_arrive_expect_tx(&bars.kfull[ks], kKTileBytes);
            tma_load_2d(kdst, &tmk, &bars.kfull[ks], w.g * kD, j0);
            tma_load_2d(kdst + kKTileBytes / 2, &tmk, &bars.kfull[ks], w.g * kD + 32, j0);
          }
          const int vs = n % kVRawStages;
          if (n >= kVRawStages && !wait_bar(&bars.vrfree[vs], ((n / kVRawStages) - 1) & 1, prm, abort_flag))
            goto producer_done;
          uint8_t* vdst = smem + kSmemVRaw + vs * kKTileBytes;
          mbar_arrive_expect_tx(&bars.vfull[vs], kKTileBytes);
          tma_load_2d(vdst, &tmv, &bars.vfull[vs], w.g * kD, j0);
          tma_load_2d(vdst + kKTileBytes / 2, &tmv, &bars.vfull[vs], w.g * kD + 32, j0);
        }
        ++lu;
      }
    producer_done:
      if (*abort_flag) {
        // Copies already issued land within microseconds; let them finish
        // before the block can exit.
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) __nanosleep(1000);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      int n = 0, lu = 0;
      auto issue_qk = [&](int m) -> bool {
        const int ks = m % kKStages;
        if (!wait_bar(&bars.kconv[ks], (m / kKStages) & 1, prm, abort_flag)) return false;
        tc_fence_after();
        const uint32_t kb = smem_u32(smem + kSmemK + ks * 2 * kKTileBytes);
        const uint32_t klo = kb + kKTileBytes;
        const uint32_t d = tmem + kColS + (m & 1) * 64;
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_tf32_ts(d, tmem + kColQhi + s * 8, sdesc_sw128(kb + (s >> 2) * 8192 + (s & 3) * 32), kIdesc, s > 0);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_tf32_ts(d, tmem + kColQhi + s * 8, sdesc_sw128(klo + (s >> 2) * 8192 + (s & 3) * 32), kIdesc, 1);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_tf32_ts(d, tmem + kColQlo + s * 8, sdesc_sw128(kb + (s >> 2) * 8192 + (s & 3) * 32), kIdesc, 1);
        mma_commit(&bars.sfull[m & 1]);
        mma_commit(&bars.kempty[ks]);
        return true;
      };
      auto issue_pv = [&](int m, bool first) -> bool {
        const int vs = m % kVStages;
        if (!wait_bar(&bars.vconv[vs], (m / kVStages) & 1, prm, abort_flag)) return false;
        tc_fence_after();
        const uint32_t vhi = smem_u32(smem + kSmemVT + vs * 2 * kKTileBytes);
        const uint32_t vlo = vhi + kKTileBytes;
        const uint32_t phi = tmem + kColS + (m & 1) * 64;
        const uint32_t plo = tmem + kColPlo + (m & 1) * 64;
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_tf32_ts(tmem + kColO, phi + s * 8, sdesc_sw128(vhi + (s >> 2) * 8192 + (s & 3) * 32), kIdesc,
                      (first && s == 0) ? 0u : 1u);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_tf32_ts(tmem + kColO, phi + s * 8, sdesc_sw128(vlo + (s >> 2) * 8192 + (s & 3) * 32), kIdesc, 1);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          mma_tf32_ts(tmem + kColO, plo + s * 8, sdesc_sw128(vhi + (s >> 2) * 8192 + (s & 3) * 32), kIdesc, 1);
        mma_commit(bars.odone);
        mma_commit(&bars.vempty[vs]);
        return true;
      };
      for (int k = 0;; ++k) {
        const int u = unit_index(k, cta, grid);
        if (u >= prm.n_units) break;
        const Unit w = decode_unit(u, prm);
        if (!wait_bar(bars.qready, lu & 1, prm, abort_flag)) goto mma_done;
        tc_fence_after();
        for (int j = 0; j < w.ntiles; ++j, ++n) {
          if (j == 0 && !issue_qk(n)) goto mma_done;
          if (j + 1 < w.ntiles && !issue_qk(n + 1)) goto mma_done;
          if (!wait_bar(&bars.pfull[n & 1], (n >> 1) & 1, prm, abort_flag)) goto mma_done;
          tc_fence_after();
          if (!issue_pv(n, j == 0)) goto mma_done;
        }
        ++lu;
      }
    mma_done:
      if (*abort_flag) {
        // Nothing may be in flight when TMEM is released.
        mma_commit(bars.drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bars.drain, 0) && globaltimer_ns() - t0 < prm.timeout_ns) {
        }
      }
    }
    __syncwarp();
  } else if (warp >= kFirstConvWarp) {
    // ----------------------------------------------------------- converters
    const int cw = warp - kFirstConvWarp;
    const int ct = threadIdx.x - kFirstConvWarp * 32;
    int n = 0;
    for (int k = 0;; ++k) {
      const int u = unit_index(k, cta, grid);
      if (u >= prm.n_units) break;
      const Unit w = decode_unit(u, prm);
      for (int j = 0; j < w.ntiles; ++j, ++n) {
        // K: lo = K - tf32_hi(K), same swizzled layout; hi in place unless the
        // tensor core truncates by itself.
        const int ks = n % kKStages;
        if (!wait_bar_warp(&bars.kfull[ks], (n / kKStages) & 1, prm, abort_flag)) goto conv_done;
        {
          uint8_t* kb = smem + kSmemK + ks * 2 * kKTileBytes;
#pragma unroll
          for (int i = 0; i < kKTileBytes / 16 / (kConvWarps * 32); ++i) {
            const uint32_t off = (uint32_t)(ct + i * kConvWarps * 32) * 16u;
            float4 x = *reinterpret_cast<const float4*>(kb + off);
            float4 hi = make_float4(tf32_hi(x.x), tf32_hi(x.y), tf32_hi(x.z), tf32_hi(x.w));
            *reinterpret_cast<float4*>(kb + kKTileBytes + off) =
                make_float4(x.x - hi.x, x.y - hi.y, x.z - hi.z, x.w - hi.w);
            if (!kHwTruncatesTf32) *reinterpret_cast<float4*>(kb + off) = hi;
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.kconv[ks]);

        // V: raw [key][d] (two d-half regions) -> V^T hi / lo [d][key] (two
        // key-half regions). Lane = key within a 32-key half; this warp takes
        // head-dimension chunks 4 cw .. 4 cw + 3.
        const int vr = n % kVRawStages;
        const int vs = n % kVStages;
        if (!wait_bar_warp(&bars.vfull[vr], (n / kVRawStages) & 1, prm, abort_flag)) goto conv_done;
        if (n >= kVStages && !wait_bar_warp(&bars.vempty[vs], ((n / kVStages) - 1) & 1, prm, abort_flag))
          goto conv_done;
        {
          const uint8_t* vraw = smem + kSmemVRaw + vr * kKTileBytes;
          uint8_t* vthi = smem + kSmemVT + vs * 2 * kKTileBytes;
          uint8_t* vtlo = vthi + kKTileBytes;
#pragma unroll
          for (int kh = 0; kh < 2; ++kh) {
            const int key = kh * 32 + lane;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int d4 = cw * 4 + c;  // 4 head dimensions 4 d4 .. 4 d4 + 3
              const float4 x = *reinterpret_cast<const float4*>(
                  vraw + (d4 >> 3) * 8192 + sw128((uint32_t)key * 128u + (uint32_t)(d4 & 7) * 16u));
              const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const uint32_t off = kh * 8192 + sw128((uint32_t)(d4 * 4 + i) * 128u + (uint32_t)lane * 4u);
                const float hi = tf32_hi(xs[i]);
                *reinterpret_cast<float*>(vthi + off) = hi;
                *reinterpret_cast<float*>(vtlo + off) = xs[i] - hi;
              }
            }
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars.vrfree[vr]);
          mbar_arrive(&bars.vconv[vs]);
        }
      }
    }
  conv_done:;
  } else {
    // -------------------------------------------------- softmax (warps 0-3)
    const int row = warp * 32 + lane;  // TMEM lane
    const uint32_t lane_tmem = tmem + ((uint32_t)(warp * 32) << 16);
    const float c = kLog2e * kScale;   // exp(s / 8) = 2^(s c)
    const float stale = kStaleLog2 / c;  // in raw-score units
    int n = 0, lu = 0;
    uint32_t od = 0;  // PV completions consumed

    // Split the unit's Q tile (staged by TMA, 128-byte swizzled) into TMEM.
    auto load_q = [&](int which) -> bool {
      if (!wait_bar_warp(bars.qfull, which & 1, prm, abort_flag)) return false;
      float hi[32], lo[32];
#pragma unroll
      for (int dh = 0; dh < 2; ++dh) {
        const uint8_t* src = smem + kSmemQ + dh * (kQBytes / 2);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float4 x = *reinterpret_cast<const float4*>(src + sw128((uint32_t)row * 128u + (uint32_t)c4 * 16u));
          const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            hi[c4 * 4 + i] = tf32_hi(xs[i]);
            lo[c4 * 4 + i] = xs[i] - hi[c4 * 4 + i];
          }
        }
        tmem_st32(lane_tmem + kColQhi + dh * 32, hi);
        tmem_st32(lane_tmem + kColQlo + dh * 32, lo);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bars.qfree);
        mbar_arrive(bars.qready);
      }
      return true;
    };

    bool q_loaded = false;
    for (int k = 0;; ++k) {
      const int u = unit_index(k, cta, grid);
      if (u >= prm.n_units) break;
      const Unit w = decode_unit(u, prm);
      if (!q_loaded && !load_q(lu)) goto softmax_done;
      q_loaded = false;
      float m_ref = -INFINITY, l = 0.f;
      const int pos = w.t0 + (row >> 2);
      const int limit = p.P + pos;  // last visible key of this row
      for (int j = 0; j < w.ntiles; ++j, ++n) {
        const int j0 = j * kBc;
        if (!wait_bar_warp(&bars.sfull[n & 1], (n >> 1) & 1, prm, abort_flag)) goto softmax_done;
        tc_fence_after();
        float s[64];
        {
          float* s0 = s;
          float* s1 = s + 32;
          tmem_ld32(lane_tmem + kColS + (n & 1) * 64, *reinterpret_cast<float(*)[32]>(s0));
          tmem_ld32(lane_tmem + kColS + (n & 1) * 64 + 32, *reinterpret_cast<float(*)[32]>(s1));
          tmem_wait_ld();
        }
        if (j0 + kBc - 1 > p.P + w.t0) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (j0 + i > limit) s[i] = -INFINITY;
        }
        float mt = s[0];
#pragma unroll
        for (int i = 1; i < 64; ++i) mt = fmaxf(mt, s[i]);
        float alpha = 1.f;
        if (m_ref == -INFINITY || mt > m_ref + stale) {
          const float m_new = fmaxf(m_ref, mt);
          alpha = (m_ref == -INFINITY) ? 0.f : ex2((m_ref - m_new) * c);
          m_ref = m_new;
        }
        const float mc = m_ref == -INFINITY ? 0.f : m_ref * c;
        float lsum = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float hi[32], lo[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float pj = ex2(fmaf(s[half * 32 + i], c, -mc));
            lsum += pj;
            hi[i] = tf32_hi(pj);
            lo[i] = pj - hi[i];
          }
          tmem_st32(lane_tmem + kColS + (n & 1) * 64 + half * 32, hi);
          tmem_st32(lane_tmem + kColPlo + (n & 1) * 64 + half * 32, lo);
        }
        l = fmaf(l, alpha, lsum);
        tmem_wait_st();
        if (j > 0) {
          // PV of the previous tile must be complete before O is touched.
          if (!wait_bar_warp(bars.odone, od & 1, prm, abort_flag)) goto softmax_done;
          ++od;
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
            float o[32];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              tmem_ld32(lane_tmem + kColO + half * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] *= alpha;
              tmem_st32(lane_tmem + kColO + half * 32, o);
            }
            tmem_wait_st();
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.pfull[n & 1]);
      }
      // The next unit's Q can go into TMEM now: its last QK has completed.
      {
        const int u_next = unit_index(k + 1, cta, grid);
        if (u_next < prm.n_units) {
          if (!load_q(lu + 1)) goto softmax_done;
          q_loaded = true;
        }
      }
      // Epilogue: wait for the last PV, one division per element.
      if (!wait_bar_warp(bars.odone, od & 1, prm, abort_flag)) goto softmax_done;
      ++od;
      tc_fence_after();
      {
        float* dst = p.out + ((size_t)pos * kHQ + w.g * kGroup + (row & 3)) * kD;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float o[32];
          tmem_ld32(lane_tmem + kColO + half * 32, o);
          tmem_wait_ld();
          if (pos < p.C) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(dst + half * 32 + i) =
                  make_float4(o[i] / l, o[i + 1] / l, o[i + 2] / l, o[i + 3] / l);
          }
        }
      }
      tc_fence_before();
      ++lu;
    }
  softmax_done:;
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

int encode_maps(const Problem& p, CUtensorMap* mq, CUtensorMap* mk, CUtensorMap* mv) {
  auto enc = get_encoder();
  if (!enc) return ATTN_ETMA;
  const cuuint32_t ones[3] = {1, 1, 1};
  // q [C][32][64] as (d, head, position); a box is 32 d x 4 heads x 32 positions.
  {
    const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)kHQ, (cuuint64_t)p.C};
    const cuuint64_t strides[2] = {(cuuint64_t)kD * 4, (cuuint64_t)kHQ * kD * 4};
    const cuuint32_t box[3] = {32, (cuuint32_t)kGroup, (cuuint32_t)kBq};
    if (enc(mq, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(p.q), dims, strides, box, ones,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return ATTN_ETMA;
  }
  // k, v [T][8][64] as (head * 64 + d, position); a box is 32 floats x 64 keys.
  const cuuint64_t T = (cuuint64_t)p.P + (cuuint64_t)p.C;
  const cuuint64_t dims[2] = {(cuuint64_t)kHKV * kD, T};
  const cuuint64_t strides[1] = {(cuuint64_t)kHKV * kD * 4};
  const cuuint32_t box[2] = {32, (cuuint32_t)kBc};
  if (enc(mk, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(p.k), dims, strides, box, ones,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return ATTN_ETMA;
  if (enc(mv, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(p.v), dims, strides, box, ones,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return ATTN_ETMA;
  return ATTN_OK;
}

struct TcDeviceState {
  bool ready = false;
  int num_sms = 0;
};
TcDeviceState g_tc_state[64];

int tc_launch_impl(const Problem& p, cudaStream_t stream, unsigned long long timeout_ns, int fault) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ECUDA;
  TcDeviceState& st = g_tc_state[dev];
  if (!st.ready) {
    if (cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTN_ECUDA;
    if (cudaFuncSetAttribute(tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc) !=
        cudaSuccess)
      return ATTN_ECUDA;
    st.ready = true;
  }
  alignas(64) CUtensorMap mq, mk, mv;
  const int rc = encode_maps(p, &mq, &mk, &mv);
  if (rc != ATTN_OK) return rc;
  Params prm;
  prm.p = p;
  prm.n_qtiles = (p.C + kBq - 1) / kBq;
  prm.n_units = prm.n_qtiles * kHKV;
  prm.timeout_ns = timeout_ns;
  prm.fault_skip_first_k = fault;
  const int grid = prm.n_units < st.num_sms ? prm.n_units : st.num_sms;
  tc_kernel<<<grid, kThreads, kSmemAlloc, stream>>>(mq, mk, mv, prm);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ELAUNCH;
}

}  // namespace

int launch_tc(const Problem& p, cudaStream_t stream) {
  return tc_launch_impl(p, stream, 2000000000ull, 0);
}

int launch_tc_fault_test(const Problem& p, cudaStream_t stream) {
  return tc_launch_impl(p, stream, 20000000ull, 1);
}

}  // namespace attn
