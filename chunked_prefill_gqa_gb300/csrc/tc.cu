// tc.cu -- the main path: persistent, warp-specialised flash prefill on the
// sm_103a tensor cores (tcgen05, TMEM accumulators, TMA staging).
//
// What it computes is the tiled online-softmax attention of "Inference
// Attention 2: Flash Prefill Against a Cached Prefix" (Lesson): a chunk of C
// rows at positions P..P+C-1 against keys 0..P+C-1, row i seeing j <= P+i,
// query head h reading KV head h/4, scale 1/8. Per tile with maximum m_tile:
// m_new = max(m_old, m_tile), alpha = exp(m_old - m_new), l and the
// accumulator rescaled by alpha, normalised by l at the very end.
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
// fp32, dropping only lo*lo (relative size 2^-20). The two terms that share
// an A operand run as one MMA of N = 128 by stacking the B operands:
//   S' = Q_hi [K_hi; K_lo]^T  (N = 128)   then  S'[:, :64] += Q_lo K_hi^T
//   S  = S'[:, :64] + S'[:, 64:]            (summed by the softmax warps)
//   O' += P_hi [V_hi V_lo]  (N = 128)     then  O'[:, :64] += P_lo V_hi
//   O  = O'[:, :64] + O'[:, 64:]            (summed in the epilogue)
// Q hi/lo and K are 128-byte-swizzled K-major shared-memory operands, V an
// MN-major one (rows are keys, as TMA lands them, swizzled in 32-byte chunks
// as MN-major 32-bit operands must be), and the tensor core reads
// raw K and V as their tf32 hi parts by itself; P is a TMEM operand (P hi and
// P lo overwrite the S columns they came from).
// TMEM holds three S buffers (QK runs up to two tiles ahead of the softmax)
// and O'.
//
// Warp roles (12 warps):
//   0-3   softmax: warp w owns TMEM lanes 32 w .. + 31 (one row per thread)
//         and all 64 keys of every tile. They split Q into shared memory at the
//         start of a unit, run the online softmax, write P hi/lo, rescale O
//         when the reference maximum moves, and write the output.
//   4     K producer: TMA loads of K tiles into the K ring.
//   5     QK issuer: allocates TMEM; one lane issues QK(n) as soon as K(n) is
//         converted and S buffer n % 3 is free (PV(n-3) complete).
//   6     V producer: TMA loads of V tiles into the V ring.
//   7-8   K converters: K lo next to each K tile (one d-half each).
//   9-10  V converters: V lo next to each V tile (one d-half each).
//   11    PV issuer: one lane issues PV(n) as soon as P(n) and V lo(n) are ready.
// The two issuers are separate threads so that neither stream of MMAs waits
// behind the other's inputs: the tensor core's issue queue is shallow, and a
// single issuer that blocks on one condition leaves the pipe idle.
// Every wait is bounded; on expiry the kernel records ATTN_ETIMEOUT in the
// device error word, all roles wind down, and TMEM is freed.
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
constexpr int kBc = 64;           // keys per tile
constexpr int kKStages = 2;       // K ring: [K | K lo] per d-half region
constexpr int kVStages = 3;       // V ring: [V | V lo], each as two d-half regions
constexpr int kNumS = 3;          // S / P buffers in TMEM

constexpr int kSoftmaxWarps = 4;
constexpr int kKProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kVProducerWarp = 6;
constexpr int kFirstKConvWarp = 7;
constexpr int kKConvWarps = 2;
constexpr int kFirstVConvWarp = 9;
constexpr int kVConvWarps = 2;
constexpr int kPvWarp = kFirstVConvWarp + kVConvWarps;
constexpr int kThreads = 32 * (kPvWarp + 1);

// TMEM columns (fp32, one per column).
constexpr uint32_t kColS = 0;    // three 128-column S buffers; P hi | P lo overwrite them
constexpr uint32_t kColO = 384;  // O' = [P_hi V_hi + P_lo V_hi | P_hi V_lo]
constexpr uint32_t kTmemCols = 512;

// Shared memory (byte offsets from a 1024-aligned base). An operand region
// is rows of 128 bytes (32 floats) in the 128-byte swizzle, 8-row groups
// 1024 bytes apart; a stacked region holds 64 hi rows then 64 lo rows.
constexpr uint32_t kRegion = 128 * 128;                  // 16 KB: 128 rows
constexpr uint32_t kHalf = 64 * 128;                     // 8 KB: 64 rows
constexpr uint32_t kKStageBytes = 2 * kRegion;           // 2 d-half regions
constexpr uint32_t kVStageBytes = 4 * kHalf;            // V d-halves 0, 1, then V lo d-halves 0, 1
constexpr uint32_t kSmemQ = 0;                           // Q hi (two d-half regions), then Q lo
constexpr uint32_t kQTermBytes = 2 * kRegion;             // 32 KB per term
constexpr uint32_t kSmemK = kSmemQ + 2 * kQTermBytes;
constexpr uint32_t kSmemV = kSmemK + kKStages * kKStageBytes;
constexpr uint32_t kSmemBar = kSmemV + kVStages * kVStageBytes;
constexpr uint32_t kNumBars = 3 * kKStages + 3 * kVStages + 3 * kNumS + 1 + 2 + 2;
constexpr uint32_t kSmemTotal = kSmemBar + kNumBars * 8 + 16;
constexpr uint32_t kSmemAlloc = kSmemTotal + 1024;  // slack to align the base

static_assert(kSmemAlloc <= 232448, "exceeds the 227 KB per-block shared memory limit");
static_assert(kM == 128 && kD == 64 && kBc == 64, "the MMA shapes below assume 128 x 64 x 64");

constexpr uint32_t kIdescN128 = idesc_tf32(128, 128);
constexpr uint32_t kIdescN64 = idesc_tf32(128, 64);
constexpr uint32_t kIdescPvN128 = idesc_tf32(128, 128, true);  // B (V) MN-major
constexpr uint32_t kIdescPvN64 = idesc_tf32(128, 64, true);
// Keep a stale reference maximum while the new maximum exceeds it by at most
// this much in log2 units (p stays <= 2^8): l and O share the reference, so
// O / l is exact either way, and O needs no rescale.
constexpr float kStaleLog2 = 8.0f;

struct Params {
  Problem p;
  int n_units;
  int n_qtiles;
  unsigned long long timeout_ns;
  int fault_skip_first_k;  // test hook: never load the first K tile
  // Paged K/V ("FlashAttention and inference kernels", PagedAttention): token t
  // lives in slot t % 16 of physical page table[t / 16]. table == nullptr:
  // contiguous [P + C][8][64] caches.
  const int* table;
  int num_pages;
  int unit_base;  // tail kernel: pair p splits unit unit_base + p
};

constexpr int kPage = 16;  // tokens per page of a paged cache

struct Bars {
  uint64_t* kfull;   // [kKStages] TMA K landed
  uint64_t* kconv;   // [kKStages] K lo written
  uint64_t* kempty;  // [kKStages] QK done with the stage (MMA commit)
  uint64_t* vfull;   // [kVStages] TMA V landed
  uint64_t* vconv;   // [kVStages] V lo written (and V rows past the sequence zeroed)
  uint64_t* vempty;  // [kVStages] PV done with the stage (MMA commit)
  uint64_t* sfull;   // [kNumS] S buffer written (MMA commit)
  uint64_t* pfull;   // [kNumS] P hi/lo written and O rescaled (softmax warps)
  uint64_t* odone;   // [kNumS] PV(n) done, barrier n % 3 (MMA commit)
  uint64_t* qready;  // Q hi/lo in shared memory (softmax warps)
  uint64_t* drain;   // [2] drain of each MMA issuer on abort (QK, PV)
  uint64_t* partner;   // tail kernel, rank 0: rank 1's share of the unit has landed (one arrival + bulk-copy bytes)
  uint64_t* slotfree;  // tail kernel, rank 1: rank 0's Q region is free for that share (128 remote arrivals)
};

__device__ __forceinline__ Bars carve_bars(uint8_t* base) {
  uint64_t* b = reinterpret_cast<uint64_t*>(base + kSmemBar);
  Bars r;
  r.kfull = b; b += kKStages;
  r.kconv = b; b += kKStages;
  r.kempty = b; b += kKStages;
  r.vfull = b; b += kVStages;
  r.vconv = b; b += kVStages;
  r.vempty = b; b += kVStages;
  r.sfull = b; b += kNumS;
  r.pfull = b; b += kNumS;
  r.odone = b; b += kNumS;
  r.qready = b++;
  r.drain = b; b += 2;
  r.partner = b++;
  r.slotfree = b++;
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

// Epilogue of a unit split over the CTA pair, for one softmax thread (row).
// Each CTA holds O (the two stacked halves of O' added), m and l of its own
// key tiles relative to its own reference maximum (none when it got no tile).
// The output is only written, never read back. Rank 1 stages its unnormalised
// O rows, m and l in its own Q region (its MMAs are complete); rank 0, once
// its last PV has completed (so its Q region is idle), tells rank 1 so, and
// each warp of rank 1 copies its 32 rows in bulk (cp.async.bulk between the
// CTAs' shared memories) into rank 0's Q region, the bytes completing on rank
// 0's partner barrier. Rank 0 then merges with the split-K rule, m = max(m0,
// m1), weights e^(m_s - m) (in log2 units, (m_s - m) c), one reciprocal of
// the merged denominator per row, and stores the row. A row is 256 bytes, its
// 16-byte chunk i at chunk i ^ (row mod 16), so the 32 rows of a warp spread
// over the banks. Measured against 16 scattered remote stores per thread:
// 247.1 against 243.6-246.0 TFLOP/s at the serving chunk. Inlined: out of
// line, the reference to the barrier set put it on the stack, and the pair
// grid measured slower.
constexpr uint32_t kShareO = 128 * 256;               // O rows, then m and l
constexpr uint32_t kShareBytes = kShareO + 2 * 128 * 4;
__device__ __forceinline__ uint32_t share_offset(int row, int i) {
  return (uint32_t)row * 256u + (uint32_t)((i ^ (row & 15)) * 16);
}

__device__ __forceinline__ bool split_epilogue(uint8_t* smem, uint32_t lane_tmem, int n, bool has, const Bars& bars,
                                               const Params& prm, volatile int* abort_flag, uint32_t rank, int row,
                                               float m_ref, float l, float c, bool store, float* dst) {
  float o[64];
  if (has) {
    const int pb = (n - 1) % kNumS;
    if (!wait_bar_warp(&bars.odone[pb], ((n - 1) / kNumS) & 1, prm, abort_flag)) return false;
    tc_fence_after();
#pragma unroll
    for (int dh = 0; dh < 2; ++dh) {
      float a[32], b[32];
      tmem_ld32(lane_tmem + kColO + dh * 32, a);
      tmem_ld32(lane_tmem + kColO + 64 + dh * 32, b);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) o[dh * 32 + i] = a[i] + b[i];
    }
  } else {
#pragma unroll
    for (int i = 0; i < 64; ++i) o[i] = 0.f;
  }
  const uint32_t peer = rank ^ 1u;
  uint8_t* share = smem + kSmemQ;
  float* ml = reinterpret_cast<float*>(share + kShareO);  // [m of the rows][l of the rows]
  if (rank == 1) {
    // Stage O, m and l in this CTA's own Q region (its MMAs are complete);
    // once rank 0's Q region is free, each warp copies its own 32 rows there
    // in bulk (O rows, m, l), completing on rank 0's partner barrier.
#pragma unroll
    for (int i = 0; i < 16; ++i)
      *reinterpret_cast<float4*>(share + share_offset(row, i)) =
          make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
    ml[row] = m_ref;
    ml[kM + row] = l;
    fence_proxy_async_smem();
    __syncwarp();
    if (!wait_bar_cluster_warp(bars.slotfree, 0, prm, abort_flag)) return false;
    if ((row & 31) == 0) {
      const uint32_t bar = mapa_shared(smem_u32(bars.partner), peer);
      const uint32_t o_off = (uint32_t)row * 256u;
      bulk_copy_to_cluster(mapa_shared(smem_u32(share + o_off), peer), share + o_off, 32 * 256, bar);
      bulk_copy_to_cluster(mapa_shared(smem_u32(ml + row), peer), ml + row, 32 * 4, bar);
      bulk_copy_to_cluster(mapa_shared(smem_u32(ml + kM + row), peer), ml + kM + row, 32 * 4, bar);
    }
  } else {
    // Every PV of this CTA is complete: its Q region may be overwritten.
    mbar_arrive_remote(mapa_shared(smem_u32(bars.slotfree), peer));
    if (row == 0) mbar_arrive_expect_tx(bars.partner, kShareBytes);
    if (!wait_bar_cluster_warp(bars.partner, 0, prm, abort_flag)) return false;
    const float m1 = ml[row], l1 = ml[kM + row];
    const float m = fmaxf(l > 0.f ? m_ref : -INFINITY, l1 > 0.f ? m1 : -INFINITY);
    const float e0 = l > 0.f ? ex2((m_ref - m) * c) : 0.f;
    const float e1 = l1 > 0.f ? ex2((m1 - m) * c) : 0.f;
    const float inv = 1.f / fmaf(e0, l, e1 * l1);  // > 0: the unit sees at least key 0
    if (store) {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 x1 = *reinterpret_cast<const float4*>(share + share_offset(row, i));
        *reinterpret_cast<float4*>(dst + 4 * i) =
            make_float4(fmaf(e0, o[4 * i], e1 * x1.x) * inv, fmaf(e0, o[4 * i + 1], e1 * x1.y) * inv,
                        fmaf(e0, o[4 * i + 2], e1 * x1.z) * inv, fmaf(e0, o[4 * i + 3], e1 * x1.w) * inv);
      }
    }
  }
  return true;
}

// The same for a unit split over a cluster of three, four, eight or twelve
// CTAs. With three or four, ranks 1.. stage their shares in their own Q
// regions and, once rank 0's last PV has completed (its Q region and K and V
// rings are then idle), copy them in bulk into consecutive slots there (rank
// r into slot r - 1). With eight, ranks 2-4 send to rank 0's slots 0-2 and
// ranks 5-7 to rank 1's; rank 1 merges its three with its own partial and
// sends that, staged in its idle V ring, to rank 0's slot 3. With twelve,
// ranks 4-11 send to ranks 0-3 two each ((r - 4) / 2, slot (r - 4) mod 2);
// ranks 1-3 merge theirs and send to rank 0's slots 2-4. A receiver merges
// its partials with the same rule: m = the largest maximum of a part with
// tiles, each part weighted by e^(m_s - m).
static_assert(kSmemQ + 5 * kShareBytes <= kSmemBar, "five shares fit in the Q region and the K and V rings");
template <int kSplit>
__device__ __forceinline__ bool split_epilogue_many(uint8_t* smem, uint32_t lane_tmem, int n, bool has,
                                                    const Bars& bars, const Params& prm, volatile int* abort_flag,
                                                    uint32_t rank, int row, float m_ref, float l, float c,
                                                    bool store, float* dst) {
  static_assert(kSplit == 3 || kSplit == 4 || kSplit == 8 || kSplit == 12, "clusters of three, four, eight or twelve");
  float o[64];
  if (has) {
    const int pb = (n - 1) % kNumS;
    if (!wait_bar_warp(&bars.odone[pb], ((n - 1) / kNumS) & 1, prm, abort_flag)) return false;
    tc_fence_after();
#pragma unroll
    for (int dh = 0; dh < 2; ++dh) {
      float a[32], b[32];
      tmem_ld32(lane_tmem + kColO + dh * 32, a);
      tmem_ld32(lane_tmem + kColO + 64 + dh * 32, b);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) o[dh * 32 + i] = a[i] + b[i];
    }
  } else {
#pragma unroll
    for (int i = 0; i < 64; ++i) o[i] = 0.f;
  }
  uint8_t* share = smem + kSmemQ;
  // Receive `nslots` shares into slots 0.. of this CTA's Q region onward from
  // `first` .. first + nslots - 1, and fold them into (o, m_ref, l): o and l
  // end up relative to the merged maximum, returned in m_ref.
  auto receive = [&](uint32_t first, int nslots) -> bool {
    for (int r = 0; r < nslots; ++r) mbar_arrive_remote(mapa_shared(smem_u32(bars.slotfree), first + (uint32_t)r));
    if (row == 0) mbar_arrive_expect_tx(bars.partner, (uint32_t)nslots * kShareBytes);
    if (!wait_bar_cluster_warp(bars.partner, 0, prm, abort_flag)) return false;
    float m = l > 0.f ? m_ref : -INFINITY;
#pragma unroll 4
    for (int r = 0; r < nslots; ++r) {
      const float* ml = reinterpret_cast<const float*>(share + r * kShareBytes + kShareO);
      if (ml[kM + row] > 0.f) m = fmaxf(m, ml[row]);
    }
    const float e0 = l > 0.f ? ex2((m_ref - m) * c) : 0.f;
    float den = e0 * l;
#pragma unroll
    for (int i = 0; i < 64; ++i) o[i] *= e0;
#pragma unroll 4
    for (int r = 0; r < nslots; ++r) {
      const uint8_t* slot = share + r * kShareBytes;
      const float* ml = reinterpret_cast<const float*>(slot + kShareO);
      const float lr = ml[kM + row];
      const float er = lr > 0.f ? ex2((ml[row] - m) * c) : 0.f;
      den = fmaf(er, lr, den);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 x = *reinterpret_cast<const float4*>(slot + share_offset(row, i));
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
  // Stage (o, m_ref, l) at `stage` in this CTA and, once the receiver says its
  // slots are free, copy each warp's 32 rows in bulk into slot `slot` of CTA
  // `to`, completing on that CTA's partner barrier.
  auto send = [&](uint8_t* stage, uint32_t to, uint32_t slot) -> bool {
    float* ml = reinterpret_cast<float*>(stage + kShareO);  // [m of the rows][l of the rows]
#pragma unroll
    for (int i = 0; i < 16; ++i)
      *reinterpret_cast<float4*>(stage + share_offset(row, i)) =
          make_float4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
    ml[row] = m_ref;
    ml[kM + row] = l;
    fence_proxy_async_smem();
    __syncwarp();
    if (!wait_bar_cluster_warp(bars.slotfree, 0, prm, abort_flag)) return false;
    if ((row & 31) == 0) {
      const uint32_t bar = mapa_shared(smem_u32(bars.partner), to);
      const uint32_t dst_slot = smem_u32(share) + slot * kShareBytes;  // the same offset in `to`
      const uint32_t o_off = (uint32_t)row * 256u;
      bulk_copy_to_cluster(mapa_shared(dst_slot + o_off, to), stage + o_off, 32 * 256, bar);
      bulk_copy_to_cluster(mapa_shared(dst_slot + kShareO + row * 4, to), ml + row, 32 * 4, bar);
      bulk_copy_to_cluster(mapa_shared(dst_slot + kShareO + (kM + row) * 4, to), ml + kM + row, 32 * 4, bar);
    }
    return true;
  };
  if (rank == 0) {
    if (!receive(1, kSplit == 12 ? 5 : kSplit == 8 ? 4 : kSplit - 1)) return false;
    const float inv = 1.f / l;  // > 0: the unit sees at least key 0
    if (store) {
#pragma unroll
      for (int i = 0; i < 16; ++i)
        *reinterpret_cast<float4*>(dst + 4 * i) =
            make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
    }
    return true;
  }
  if constexpr (kSplit == 12) {
    if (rank <= 3) {
      if (!receive(2 * rank + 4, 2)) return false;
      return send(smem + kSmemV, 0, rank + 1);
    }
    return send(share, (rank - 4) >> 1, (rank - 4) & 1);
  } else if constexpr (kSplit == 8) {
    if (rank == 1) {
      if (!receive(5, 3)) return false;
      return send(smem + kSmemV, 0, 3);
    }
    return rank < 5 ? send(share, 0, rank - 2) : send(share, 1, rank - 5);
  } else {
    return send(share, 0, rank - 1);
  }
}

// Instantiations. kMain: whole units in snake order; it decides by prm.table
// at run time (it is the one launched for contiguous caches; measured,
// dropping its paged branch slows it). kPaged: the same for page pools only.
// kTail: launched after kMain as clusters of two CTAs; pair p splits unit
// unit_base + p along its key tiles (rank 0 the first half, rank 1 the rest)
// and merges the two online-softmax partials through distributed shared memory.
// kTail3, kTail4, kTail8, kTail12: the same with clusters of three, four,
// eight or twelve CTAs, each that share of the unit's tiles (small chunks,
// whose units are too few to fill the SMs as pairs).
constexpr int kMain = 0, kPaged = 1, kTail = 2, kTail4 = 3, kTail8 = 4, kTail3 = 5, kTail12 = 6;
template <int kMode>
__host__ __device__ constexpr int split_of() {
  return kMode == kTail     ? 2
         : kMode == kTail3  ? 3
         : kMode == kTail4  ? 4
         : kMode == kTail8  ? 8
         : kMode == kTail12 ? 12
                            : 1;
}
template <int kMode>
__host__ __device__ constexpr bool is_tail() { return split_of<kMode>() > 1; }

// Unit u's tiles for this CTA: all of them, or the tail kernel's half.
template <int kMode>
__device__ __forceinline__ void unit_range(const Unit& w, uint32_t rank, int* jb, int* je) {
  if constexpr (kMode == kTail) {
    *jb = rank == 0 ? 0 : w.ntiles / 2;
    *je = rank == 0 ? w.ntiles / 2 : w.ntiles;
  } else if constexpr (is_tail<kMode>()) {
    constexpr int kS = split_of<kMode>();
    *jb = (int)rank * w.ntiles / kS;
    *je = ((int)rank + 1) * w.ntiles / kS;
  } else {
    *jb = 0;
    *je = w.ntiles;
  }
}

// The CTA's k-th unit (kMain, kPaged: snake order; the tail modes: one per
// cluster), or n_units when it has none.
template <int kMode>
__device__ __forceinline__ int work_unit(int k, int cta, int grid, const Params& prm) {
  if constexpr (kMode == kTail) return k == 0 ? prm.unit_base + (cta >> 1) : prm.n_units;
  else if constexpr (kMode == kTail4) return k == 0 ? prm.unit_base + (cta >> 2) : prm.n_units;
  else if constexpr (kMode == kTail8) return k == 0 ? prm.unit_base + (cta >> 3) : prm.n_units;
  else if constexpr (kMode == kTail3) return k == 0 ? prm.unit_base + cta / 3 : prm.n_units;
  else if constexpr (kMode == kTail12) return k == 0 ? prm.unit_base + cta / 12 : prm.n_units;
  else return unit_index(k, cta, grid);
}

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
          const __grid_constant__ Params prm) {
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
      mbar_init(&bars.kconv[s], kKConvWarps);
      mbar_init(&bars.kempty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&bars.vfull[s], 1);
      mbar_init(&bars.vconv[s], kVConvWarps);
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
    if constexpr (is_tail<kMode>()) {
      mbar_init(bars.partner, 1);
      mbar_init(bars.slotfree, kSoftmaxWarps * 32);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kKProducerWarp && lane == 0) tma_prefetch_desc(&tmk);
  if (warp == kVProducerWarp && lane == 0) tma_prefetch_desc(&tmv);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  if constexpr (is_tail<kMode>()) {
    // Every CTA of the cluster is running and its barriers initialised before
    // any can touch another's shared memory.
    cluster_sync_all();
  } else {
    // A tail launch after this one (a programmatic dependent) may start its
    // blocks on SMs as soon as blocks of this grid leave them.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }
  const uint32_t rank = is_tail<kMode>() ? cluster_ctarank() : 0u;

  const int cta = blockIdx.x, grid = gridDim.x;
  const Problem& p = prm.p;

  if (warp == kKProducerWarp || warp == kVProducerWarp) {
    // ------------------------------------------------------------ producers
    const bool is_k = warp == kKProducerWarp;
    // Page pools: lanes 0-3 each issue one page of a tile (its table entry and
    // its two boxes); otherwise lane 0 issues the whole tile.
    constexpr int kLanes = kMode == kPaged ? kBc / kPage : 1;
    if (lane < kLanes) {
      const int stages = is_k ? kKStages : kVStages;
      int n = 0;
      for (int k = 0;; ++k) {
        const int u = work_unit<kMode>(k, cta, grid, prm);
        if (u >= prm.n_units) break;
        const Unit w = decode_unit(u, prm);
        int jb, je;
        unit_range<kMode>(w, rank, &jb, &je);
        for (int j = jb; j < je; ++j, ++n) {
          const int st = n % stages;
          uint64_t* freed = is_k ? &bars.kempty[st] : &bars.vempty[st];
          // Page pools: each lane's block-table entry is read before the wait
          // for the stage, so its latency passes while the stage drains.
          const int lp = j * (kBc / kPage) + lane;
          int phys = 0;
          if (kMode == kPaged && lp * kPage < p.P + p.C) phys = __ldg(prm.table + lp);
          if constexpr (kMode == kPaged) {
            // The four lanes leave together or not at all.
            const bool ok = n < stages || wait_bar(freed, ((n / stages) - 1) & 1, prm, abort_flag);
            if (!__all_sync((1u << kLanes) - 1, ok)) goto producer_done;
          } else {
            if (n >= stages && !wait_bar(freed, ((n / stages) - 1) & 1, prm, abort_flag)) goto producer_done;
          }
          if (is_k && prm.fault_skip_first_k && n == 0) continue;
          const CUtensorMap* map = is_k ? &tmk : &tmv;
          uint64_t* full = is_k ? &bars.kfull[st] : &bars.vfull[st];
          uint8_t* dst = is_k ? smem + kSmemK + st * kKStageBytes : smem + kSmemV + st * kVStageBytes;
          const uint32_t half_stride = is_k ? kRegion : kHalf;  // d-half regions
          if constexpr (kMode == kPaged) {
            // Lane 0 posts the tile's bytes before any of its boxes is issued.
            if (lane == 0) mbar_arrive_expect_tx(full, 2 * kHalf);
            __syncwarp((1u << kLanes) - 1);
            int y = prm.num_pages * kPage;
            if (lp * kPage < p.P + p.C) {
              if (phys >= 0 && phys < prm.num_pages)
                y = phys * kPage;
              else
                record_error(p.err, kDevErrBounds);
            }
            tma_load_2d(dst + lane * kPage * 128, map, full, w.g * kD, y);
            tma_load_2d(dst + half_stride + lane * kPage * 128, map, full, w.g * kD + 32, y);
            continue;
          }
          mbar_arrive_expect_tx(full, 2 * kHalf);
          if (prm.table == nullptr) {
            tma_load_2d(dst, map, full, w.g * kD, j * kBc);
            tma_load_2d(dst + half_stride, map, full, w.g * kD + 32, j * kBc);
          } else {
            // Four 16-row boxes per d-half; each is two whole 1024-byte swizzle
            // atoms, so the tile lands exactly as a contiguous load would.
            // A page past the sequence, or a table entry outside [0,
            // num_pages) (also recorded as a bounds error), is read from an
            // out-of-range row, which TMA fills with zeros.
            const int T = p.P + p.C;
#pragma unroll
            for (int pg = 0; pg < kBc / kPage; ++pg) {
              const int lp = j * (kBc / kPage) + pg;
              int y = prm.num_pages * kPage;
              if (lp * kPage < T) {
                const int phys = __ldg(prm.table + lp);
                if (phys >= 0 && phys < prm.num_pages)
                  y = phys * kPage;
                else
                  record_error(p.err, kDevErrBounds);
              }
              tma_load_2d(dst + pg * kPage * 128, map, full, w.g * kD, y);
              tma_load_2d(dst + half_stride + pg * kPage * 128, map, full, w.g * kD + 32, y);
            }
          }
        }
      }
    producer_done:
      if (*abort_flag) {
        // Copies already issued land within microseconds; let them finish
        // before the block can exit.
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 200000ull) __nanosleep(1000);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp || warp == kPvWarp) {
    // ---------------------------------------------------------- MMA issuers
    const bool is_qk = warp == kMmaWarp;
    if (lane == 0) {
      int n = 0, lu = 0;
      for (int k = 0;; ++k) {
        const int u = work_unit<kMode>(k, cta, grid, prm);
        if (u >= prm.n_units) break;
        const Unit w = decode_unit(u, prm);
        int jb, je;
        unit_range<kMode>(w, rank, &jb, &je);
        if constexpr (is_tail<kMode>()) {
          if (jb == je) continue;  // no tiles here (its Q is not loaded either)
        }
        if (is_qk) {
          if (!wait_bar(bars.qready, lu & 1, prm, abort_flag)) goto mma_done;
          tc_fence_after();
        }
        for (int j = jb; j < je; ++j, ++n) {
          if (is_qk) {
            // QK(n): K(n) converted; S buffer n % 3 free once PV(n-3) has read
            // P(n-3) from it (odone[n % 3] is at most one phase past PV(n-3):
            // PV(n) needs S(n), which is issued only below).
            const int ks = n % kKStages;
            const int sb = n % kNumS;
            if (!wait_bar(&bars.kconv[ks], (n / kKStages) & 1, prm, abort_flag)) goto mma_done;
            if (n >= kNumS && !wait_bar(&bars.odone[sb], ((n / kNumS) - 1) & 1, prm, abort_flag)) goto mma_done;
            tc_fence_after();
            const uint32_t kb = smem_u32(smem + kSmemK + ks * kKStageBytes);
            const uint32_t qb = smem_u32(smem + kSmemQ);
            const uint32_t d = tmem + kColS + sb * 128;
#pragma unroll
            for (int s = 0; s < 8; ++s)  // [Q_hi K_hi^T | Q_hi K_lo^T]
              mma_tf32_ss(d, sdesc_sw128(qb + (s >> 2) * kRegion + (s & 3) * 32),
                          sdesc_sw128(kb + (s >> 2) * kRegion + (s & 3) * 32), kIdescN128, s > 0);
#pragma unroll
            for (int s = 0; s < 8; ++s)  // += Q_lo K_hi^T into the first half
              mma_tf32_ss(d, sdesc_sw128(qb + kQTermBytes + (s >> 2) * kRegion + (s & 3) * 32),
                          sdesc_sw128(kb + (s >> 2) * kRegion + (s & 3) * 32), kIdescN64, 1);
            mma_commit(&bars.sfull[sb]);
            mma_commit(&bars.kempty[ks]);
          } else {
            // PV(n): P(n) written by the softmax warps, V lo(n) written.
            // Keys 8s .. 8s + 7 are rows 8s .. 8s + 7 (one 1024-byte atom)
            // of each 8 KB d-half region; the regions in stage order (V 0-31,
            // V 32-63, V lo 0-31, V lo 32-63) are the B operand's N blocks.
            const int vs = n % kVStages;
            const int sb = n % kNumS;
            if (!wait_bar(&bars.pfull[sb], (n / kNumS) & 1, prm, abort_flag)) goto mma_done;
            if (!wait_bar(&bars.vconv[vs], (n / kVStages) & 1, prm, abort_flag)) goto mma_done;
            tc_fence_after();
            const uint32_t vb = smem_u32(smem + kSmemV + vs * kVStageBytes);
            const uint32_t phi = tmem + kColS + sb * 128;
            const uint32_t plo = phi + 64;
            const bool first = j == jb;
#pragma unroll
            for (int s = 0; s < 8; ++s)  // [P_hi V_hi | P_hi V_lo]
              mma_tf32_ts(tmem + kColO, phi + s * 8, sdesc_sw128a32_mn(vb + s * 1024, kHalf), kIdescPvN128,
                          (first && s == 0) ? 0u : 1u);
#pragma unroll
            for (int s = 0; s < 8; ++s)  // += P_lo V_hi into the first half
              mma_tf32_ts(tmem + kColO, plo + s * 8, sdesc_sw128a32_mn(vb + s * 1024, kHalf), kIdescPvN64, 1);
            mma_commit(&bars.odone[sb]);
            mma_commit(&bars.vempty[vs]);
          }
        }
        ++lu;
      }
    mma_done:
      if (*abort_flag) {
        // Nothing this thread issued may be in flight when TMEM is released.
        uint64_t* drain = &bars.drain[is_qk ? 0 : 1];
        mma_commit(drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < prm.timeout_ns) {
        }
      }
    }
    __syncwarp();
  } else if (warp >= kFirstKConvWarp && warp < kFirstKConvWarp + kKConvWarps) {
    // ---------------------------------------------------------- K converters
    // K lo = K - tf32_hi(K) into the lower half of each d-half region; warp
    // kc takes region kc. The tensor core reads raw K as tf32_hi(K) by itself:
    // it ignores the 13 low mantissa bits of an fp32 operand (measured on
    // GB300: 1 + 3 * 2^-12 reads as 1 from shared memory and from TMEM).
    const int kc = warp - kFirstKConvWarp;
    int n = 0;
    for (int k = 0;; ++k) {
      const int u = work_unit<kMode>(k, cta, grid, prm);
      if (u >= prm.n_units) break;
      const Unit w = decode_unit(u, prm);
      int jb, je;
      unit_range<kMode>(w, rank, &jb, &je);
      for (int j = jb; j < je; ++j, ++n) {
        const int ks = n % kKStages;
        if (!wait_bar_warp(&bars.kfull[ks], (n / kKStages) & 1, prm, abort_flag)) goto kconv_done;
        uint8_t* kb = smem + kSmemK + ks * kKStageBytes + kc * kRegion;
        float4 x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = *reinterpret_cast<const float4*>(kb + (uint32_t)(lane + 32 * i) * 16u);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          *reinterpret_cast<float4*>(kb + (uint32_t)(lane + 32 * i) * 16u + kHalf) =
              make_float4(x[i].x - tf32_hi(x[i].x), x[i].y - tf32_hi(x[i].y), x[i].z - tf32_hi(x[i].z),
                          x[i].w - tf32_hi(x[i].w));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.kconv[ks]);
      }
    }
  kconv_done:;
  } else if (warp >= kFirstVConvWarp) {
    // ---------------------------------------------------------- V converters
    // V lo = V - tf32_hi(V) into the stage's second half; warp cw takes d-half
    // cw. In a tile that reaches past the sequence, the rows of keys at or
    // past P + C are zeroed first, in V and V lo: they carry zero weight, but
    // 0 * NaN is NaN and the unused slots of a cache page need not hold finite
    // values. (A row of the swizzled region is one key: the swizzle only
    // permutes the 16-byte chunks within it.)
    const int cw = warp - kFirstVConvWarp;
    int n = 0;
    for (int k = 0;; ++k) {
      const int u = work_unit<kMode>(k, cta, grid, prm);
      if (u >= prm.n_units) break;
      const Unit w = decode_unit(u, prm);
      int jb, je;
      unit_range<kMode>(w, rank, &jb, &je);
      for (int j = jb; j < je; ++j, ++n) {
        const int vs = n % kVStages;
        if (!wait_bar_warp(&bars.vfull[vs], (n / kVStages) & 1, prm, abort_flag)) goto vconv_done;
        uint8_t* vb = smem + kSmemV + vs * kVStageBytes + cw * kHalf;
        float4 x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = *reinterpret_cast<const float4*>(vb + (uint32_t)(lane + 32 * i) * 16u);
        if ((j + 1) * kBc > p.P + p.C) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            if (j * kBc + ((lane + 32 * i) >> 3) >= p.P + p.C) {
              x[i] = make_float4(0.f, 0.f, 0.f, 0.f);
              *reinterpret_cast<float4*>(vb + (uint32_t)(lane + 32 * i) * 16u) = x[i];
            }
          }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
          *reinterpret_cast<float4*>(vb + (uint32_t)(lane + 32 * i) * 16u + 2 * kHalf) =
              make_float4(x[i].x - tf32_hi(x[i].x), x[i].y - tf32_hi(x[i].y), x[i].z - tf32_hi(x[i].z),
                          x[i].w - tf32_hi(x[i].w));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.vconv[vs]);
      }
    }
  vconv_done:;
  } else {
    // -------------------------------------------------- softmax (warps 0-3)
    const int rq = warp;               // TMEM lanes 32 rq .. 32 rq + 31
    const int row = rq * 32 + lane;    // TMEM lane = row of the unit
    const uint32_t lane_tmem = tmem + ((uint32_t)(rq * 32) << 16);
    const float c = kLog2e * kScale;     // exp(s / 8) = 2^(s c)
    const float stale = kStaleLog2 / c;  // in raw-score units
    int n = 0;

    // The row's query (zeros past the chunk), split into tf32 hi and lo and
    // written to the two Q operand regions of shared memory, row `row`, under
    // the 128-byte swizzle (a quarter-warp's 16-byte stores fall in 8
    // distinct bank groups).
    auto load_q = [&](const Unit& w) {
      const int pos = w.t0 + (row >> 2);
      const float* src = p.q + ((size_t)pos * kHQ + w.g * kGroup + (row & 3)) * kD;
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (pos < p.C) v = __ldg(reinterpret_cast<const float4*>(src + h * 32 + c4 * 4));
          const float4 hi = make_float4(tf32_hi(v.x), tf32_hi(v.y), tf32_hi(v.z), tf32_hi(v.w));
          const uint32_t off = (uint32_t)h * kRegion + sw128((uint32_t)row * 128u + (uint32_t)c4 * 16u);
          *reinterpret_cast<float4*>(smem + kSmemQ + off) = hi;
          *reinterpret_cast<float4*>(smem + kSmemQ + kQTermBytes + off) =
              make_float4(v.x - hi.x, v.y - hi.y, v.z - hi.z, v.w - hi.w);
        }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bars.qready);
    };

    bool q_loaded = false;
    for (int k = 0;; ++k) {
      const int u = work_unit<kMode>(k, cta, grid, prm);
      if (u >= prm.n_units) break;
      const Unit w = decode_unit(u, prm);
      int jb, je;
      unit_range<kMode>(w, rank, &jb, &je);
      const bool has = jb < je;
      if (has && !q_loaded) load_q(w);
      q_loaded = false;
      float m_ref = -INFINITY, l = 0.f;
      const int pos = w.t0 + (row >> 2);
      const int limit = p.P + pos;  // last visible key of this row
      for (int j = jb; j < je; ++j, ++n) {
        const int j0 = j * kBc;
        const int sb = n % kNumS;
        const uint32_t sbuf = lane_tmem + kColS + sb * 128;
        if (!wait_bar_warp(&bars.sfull[sb], (n / kNumS) & 1, prm, abort_flag)) goto softmax_done;
        tc_fence_after();
        // S = S'[:, 0:64] + S'[:, 64:128] for the tile's 64 keys.
        float s[64];
        tmem_ld32(sbuf, *reinterpret_cast<float(*)[32]>(&s[0]));
        tmem_ld32(sbuf + 32, *reinterpret_cast<float(*)[32]>(&s[32]));
        tmem_wait_ld();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          float t[32];
          tmem_ld32(sbuf + 64 + half * 32, t);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            add2(s[half * 32 + i], s[half * 32 + i + 1], s[half * 32 + i], s[half * 32 + i + 1], t[i], t[i + 1]);
        }
        if (j0 + kBc - 1 > p.P + w.t0) {
#pragma unroll
          for (int i = 0; i < 64; ++i)
            if (j0 + i > limit) s[i] = -INFINITY;
        }
        float mt = max3(s[0], s[1], s[2]);
#pragma unroll
        for (int i = 3; i < 63; i += 2) mt = max3(mt, s[i], s[i + 1]);
        mt = fmaxf(mt, s[63]);
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
          float hi[32], lo[32];
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            float a0, a1;
            fma2(a0, a1, s[half * 32 + i], s[half * 32 + i + 1], c, c, -mc, -mc);
            const float p0 = ex2(a0), p1 = ex2(a1);
            add2(l0, l1, l0, l1, p0, p1);
            hi[i] = tf32_hi(p0);
            hi[i + 1] = tf32_hi(p1);
            fma2(lo[i], lo[i + 1], hi[i], hi[i + 1], -1.f, -1.f, p0, p1);  // p - hi, exact
          }
          tmem_st32(sbuf + half * 32, hi);
          tmem_st32(sbuf + 64 + half * 32, lo);
        }
        l = fmaf(l, alpha, l0 + l1);
        tmem_wait_st();
        // O is rescaled only when the reference maximum moved; PV(n-1) must be
        // complete first. Skipping this wait otherwise is safe for the parity
        // bookkeeping: PV(n+2) cannot run before these warps release P(n+2), so
        // odone[(n-1) % 3] is at most one phase past the one waited for here.
        if (j > jb && __any_sync(0xffffffffu, alpha != 1.f)) {
          const int pb = (n - 1) % kNumS;
          if (!wait_bar_warp(&bars.odone[pb], ((n - 1) / kNumS) & 1, prm, abort_flag)) goto softmax_done;
          tc_fence_after();
#pragma unroll
          for (int part = 0; part < 4; ++part) {  // O' columns 32 part .. + 31
            float o[32];
            tmem_ld32(lane_tmem + kColO + part * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(lane_tmem + kColO + part * 32, o);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.pfull[sb]);
      }
      // The next unit's Q can go into shared memory now: its last QK has
      // completed (its S was just consumed).
      {
        const int u_next = work_unit<kMode>(k + 1, cta, grid, prm);
        if (u_next < prm.n_units) {
          load_q(decode_unit(u_next, prm));
          q_loaded = true;
        }
      }
      if constexpr (kMode == kTail) {
        float* dst = p.out + ((size_t)pos * kHQ + w.g * kGroup + (row & 3)) * kD;
        if (!split_epilogue(smem, lane_tmem, n, has, bars, prm, abort_flag, rank, row, m_ref, l, c, pos < p.C,
                            dst))
          goto softmax_done;
        tc_fence_before();
        continue;
      } else if constexpr (is_tail<kMode>()) {
        float* dst = p.out + ((size_t)pos * kHQ + w.g * kGroup + (row & 3)) * kD;
        if (!split_epilogue_many<split_of<kMode>()>(smem, lane_tmem, n, has, bars, prm, abort_flag, rank, row,
                                                          m_ref, l, c, pos < p.C, dst))
          goto softmax_done;
        tc_fence_before();
        continue;
      }
      // Epilogue: wait for the last PV, add the two stacked halves of O' and
      // normalise by the row's l: one reciprocal per row and a multiply per
      // element, measured faster than 64 IEEE divisions per thread, except in
      // the page-pool instantiation, whose code measured faster keeping the
      // divisions (with the reciprocal it lost 4-9 %).
      {
        const int pb = (n - 1) % kNumS;
        if (!wait_bar_warp(&bars.odone[pb], ((n - 1) / kNumS) & 1, prm, abort_flag)) goto softmax_done;
      }
      tc_fence_after();
      const float norm = kMode == kPaged ? l : 1.f / l;
#pragma unroll
      for (int dh = 0; dh < 2; ++dh) {
        float a[32], b[32];
        tmem_ld32(lane_tmem + kColO + dh * 32, a);
        tmem_ld32(lane_tmem + kColO + 64 + dh * 32, b);
        tmem_wait_ld();
        if (pos < p.C) {
          float* dst = p.out + ((size_t)pos * kHQ + w.g * kGroup + (row & 3)) * kD + dh * 32;
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + i) =
                kMode == kPaged
                    ? make_float4((a[i] + b[i]) / norm, (a[i + 1] + b[i + 1]) / norm, (a[i + 2] + b[i + 2]) / norm,
                                  (a[i + 3] + b[i + 3]) / norm)
                    : make_float4((a[i] + b[i]) * norm, (a[i + 1] + b[i + 1]) * norm, (a[i + 2] + b[i + 2]) * norm,
                                  (a[i + 3] + b[i + 3]) * norm);
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
  if constexpr (is_tail<kMode>()) {
    // No CTA of the cluster leaves while another may still write its shared
    // memory or arrive on its barriers.
    cluster_sync_all();
  }
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  if constexpr (is_tail<kMode>()) {
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
PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
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

// k, v [rows][8][64] as a 2-D tensor (head * 64 + d, row); a box is 32 floats
// (one 128-byte swizzle row) x box_rows rows: 64 keys of a contiguous cache, or
// one 16-token page of a paged cache ([pages * 16][8][64]).
// K lands in the 128-byte swizzle of K-major operands; V, an MN-major tf32
// operand, in the 128-byte swizzle of 32-byte chunks that the tensor core
// requires of MN-major 32-bit operands.
int encode_kv_map(const float* base, int rows, int box_rows, CUtensorMapSwizzle swizzle, CUtensorMap* map) {
  auto enc = get_encoder();
  if (!enc) return ATTN_ETMA;
  const cuuint32_t ones[2] = {1, 1};
  const cuuint64_t dims[2] = {(cuuint64_t)kHKV * kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kHKV * kD * 4};
  const cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
  if (enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, ones,
          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return ATTN_ETMA;
  return ATTN_OK;
}

struct TcDeviceState {
  bool ready = false;
  int num_sms = 0;
  int quads = 0;   // clusters of four tail CTAs the device holds at once
  int octets = 0;  // clusters of eight
  int trios = 0;   // clusters of three
  int twelves = 0;  // clusters of twelve
};
TcDeviceState g_tc_state[64];
std::mutex g_tc_state_mu;

int tc_launch_impl(const Problem& p, cudaStream_t stream, unsigned long long timeout_ns, int fault,
                   const int* table = nullptr, int num_pages = 0) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ECUDA;
  int num_sms = 0, quads = 0, octets = 0, trios = 0, twelves = 0;
  {
    std::lock_guard<std::mutex> lock(g_tc_state_mu);
    TcDeviceState& st = g_tc_state[dev];
    if (!st.ready) {
      if (cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return ATTN_ECUDA;
      if (cudaFuncSetAttribute(tc_kernel<kMain>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc) !=
              cudaSuccess ||
          cudaFuncSetAttribute(tc_kernel<kPaged>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc) !=
              cudaSuccess ||
          cudaFuncSetAttribute(tc_kernel<kTail>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc) !=
              cudaSuccess ||
          cudaFuncSetAttribute(tc_kernel<kTail4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc) !=
              cudaSuccess ||
          cudaFuncSetAttribute(tc_kernel<kTail8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc) !=
              cudaSuccess ||
          cudaFuncSetAttribute(tc_kernel<kTail3>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc) !=
              cudaSuccess ||
          cudaFuncSetAttribute(tc_kernel<kTail12>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemAlloc) !=
              cudaSuccess)
        return ATTN_ECUDA;
      // Clusters of twelve are a non-portable size: allowed per kernel (on
      // a device that refuses, no twelve-way split).
      const bool twelve_ok =
          cudaFuncSetAttribute(tc_kernel<kTail12>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
      if (!twelve_ok) (void)cudaGetLastError();
      // How many clusters of three, four and eight fit at once (0 when a
      // query fails: no such split then).
      auto clusters_of = [&](int size, void (*kernel)(CUtensorMap, CUtensorMap, Params)) {
        cudaLaunchConfig_t qc = {};
        qc.gridDim = dim3(size * kHKV);
        qc.blockDim = dim3(kThreads);
        qc.dynamicSmemBytes = kSmemAlloc;
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
      st.quads = clusters_of(4, tc_kernel<kTail4>);
      st.octets = clusters_of(8, tc_kernel<kTail8>);
      st.trios = clusters_of(3, tc_kernel<kTail3>);
      st.twelves = twelve_ok ? clusters_of(12, tc_kernel<kTail12>) : 0;
      st.ready = true;
    }
    num_sms = st.num_sms;
    quads = st.quads;
    octets = st.octets;
    trios = st.trios;
    twelves = st.twelves;
  }
  alignas(64) CUtensorMap mk, mv;
  const int rows = table ? num_pages * kPage : p.P + p.C;
  const int box_rows = table ? kPage : kBc;
  int rc = encode_kv_map(p.k, rows, box_rows, CU_TENSOR_MAP_SWIZZLE_128B, &mk);
  if (rc == ATTN_OK) rc = encode_kv_map(p.v, rows, box_rows, CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B, &mv);
  if (rc != ATTN_OK) return rc;
  Params prm;
  prm.p = p;
  prm.n_qtiles = (p.C + kBq - 1) / kBq;
  prm.n_units = prm.n_qtiles * kHKV;
  prm.timeout_ns = timeout_ns;
  prm.fault_skip_first_k = fault;
  prm.table = table;
  prm.num_pages = num_pages;
  prm.unit_base = 0;
  const int grid = prm.n_units < num_sms ? prm.n_units : num_sms;
  // Split units. With several rounds, when the last round of whole units would
  // leave more than half of the SMs idle, the full rounds run as one grid and
  // the remaining units as a second grid of CTA pairs that each split one unit.
  // With at most half as many units as SMs and the longest unit of 256 keys or
  // more, every unit is split over a pair (with the bulk-copy hand-off,
  // measured 1.1-1.3x faster for chunks against 500-2000 keys; from 2048 keys
  // it already was; 1.1x against 250-500 keys), over a cluster of four when
  // the device holds one for every unit (chunks of 128 rows or less on 152
  // SMs: measured 1.4-1.9x faster than pairs against 2000-32768 keys, 1.1-1.2x
  // against 600-1500), and over a cluster of eight when it holds one of those
  // for every unit and the longest unit sees 1024 keys or more (15 on a GB300:
  // chunks of 32 rows or less, 1.7x faster than fours against 32768 keys), or
  // of twelve (a non-portable size, 8 on a GB300) when the longest unit sees
  // 8192 keys or more (1.1-1.3x faster than eights against 8192-32768 keys,
  // slower against 1600-2048; 16 units, more than the clusters of eight it
  // holds, go to twelves in two waves from 16384 keys: 1.07-1.18x faster than
  // fours, slower against 8192),
  // and over a cluster of three when it holds one of those for every unit
  // (46: chunks of 129-184 rows, 1.2-1.4x faster than pairs against 3000-32768
  // keys).
  // (The two grids can also split only the longest s units, the whole-unit
  // grid starting s / 8 q-tiles down.) The pair grid is a programmatic
  // dependent of the whole-unit grid: its pairs take SMs as soon as they are
  // free.
  Params main_prm = prm, tail_prm = prm;
  int main_grid = grid, tail_units = 0, split = 2;
  if (prm.n_units > grid) {
    // (Only when even the shortest unit sees 1024 keys: measured, a full
    // prompt's last round of 32-224 keys runs slower split.)
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
      else if (rem <= octets && unit_keys(p.P, p.C, 0, kBq) >= 1024)
        split = 8;
      else if (rem <= quads)
        split = 4;
      else if (rem <= trios)
        split = 3;
    } else if (rem > num_sms / 2 && rem <= 2 * trios && unit_keys(p.P, p.C, 0, kBq) >= 8192) {
      // A last round of more than half as many units as SMs: over clusters of
      // three in two waves, when its units are long (measured 1.06-1.16x for
      // chunks of 928-1568 rows against 8192-30000 keys; 0.91-1.03x against
      // 2048-4096).
      main_prm.n_units = full;
      tail_prm.unit_base = full;
      tail_units = rem;
      split = 3;
    }
  } else if (2 * prm.n_units <= num_sms && unit_keys(p.P, p.C, (prm.n_qtiles - 1) * kBq, kBq) >= 256) {
    // Measured: splitting only some of the units (more than half as many
    // units as SMs) costs more than it gains.
    main_prm.n_units = 0;
    tail_prm.unit_base = 0;
    tail_units = prm.n_units;
    if (prm.n_units <= twelves && unit_keys(p.P, p.C, (prm.n_qtiles - 1) * kBq, kBq) >= 8192)
      split = 12;
    else if (prm.n_units <= octets && unit_keys(p.P, p.C, (prm.n_qtiles - 1) * kBq, kBq) >= 1024)
      split = 8;
    else if (prm.n_units <= 2 * twelves && unit_keys(p.P, p.C, (prm.n_qtiles - 1) * kBq, kBq) >= 16384)
      split = 12;  // more units than clusters of eight: twelves in two waves (long units only)
    else if (prm.n_units <= quads)
      split = 4;
    else if (prm.n_units <= trios)
      split = 3;
  } else if (prm.n_units <= 2 * trios && unit_keys(p.P, p.C, (prm.n_qtiles - 1) * kBq, kBq) >= 4096) {
    // A partial round of more than half as many units as SMs: every unit over
    // a cluster of three, the clusters running in two waves as the device
    // frees SMs (measured 1.1-1.4x for chunks of 300-352 rows against
    // 4096-32768 keys, paged 1.1-1.2x; below that many keys, or with more
    // units, whole units stay faster).
    main_prm.n_units = 0;
    tail_prm.unit_base = 0;
    tail_units = prm.n_units;
    split = 3;
  }
  if (main_prm.n_units > 0) {
    if (table)
      tc_kernel<kPaged><<<main_grid, kThreads, kSmemAlloc, stream>>>(mk, mv, main_prm);
    else
      tc_kernel<kMain><<<main_grid, kThreads, kSmemAlloc, stream>>>(mk, mv, main_prm);
    if (cudaGetLastError() != cudaSuccess) return ATTN_ELAUNCH;
  }
  if (tail_units == 0) return ATTN_OK;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(split * tail_units);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemAlloc;
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
  auto* tail = split == 8   ? tc_kernel<kTail8>
               : split == 4 ? tc_kernel<kTail4>
               : split == 3 ? tc_kernel<kTail3>
               : split == 12 ? tc_kernel<kTail12>
                            : tc_kernel<kTail>;
  if (cudaLaunchKernelEx(&cfg, tail, mk, mv, tail_prm) != cudaSuccess) return ATTN_ELAUNCH;
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ELAUNCH;
}

}  // namespace

int launch_tc(const Problem& p, cudaStream_t stream) {
  return tc_launch_impl(p, stream, 2000000000ull, 0);
}

int launch_tc_fault_test(const Problem& p, cudaStream_t stream) {
  return tc_launch_impl(p, stream, 20000000ull, 1);
}

int launch_tc_paged(const Problem& p, const int* table, int num_pages, cudaStream_t stream) {
  return tc_launch_impl(p, stream, 2000000000ull, 0, table, num_pages);
}

}  // namespace attn
