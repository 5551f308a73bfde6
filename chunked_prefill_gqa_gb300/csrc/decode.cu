// decode.cu -- grouped-query decode against a paged K/V cache, split over the
// key range and merged with the online-softmax rule.
//
// Decode is the chunk of one token ("Inference Attention 2: Flash Prefill
// Against a Cached Prefix", Lesson: shrink the chunk to one token and the
// kernel is bandwidth-bound). Each sequence b has one query per head,
// q[b][h][:], whose key/value are already in the cache at position ctx_b - 1,
// so it attends to every cached key 0 .. ctx_b - 1.
//
// Split kernel: a block owns (segment s, KV head g, sequence b) and all four
// query heads that read g, so each K/V row is read once for the group ("FlashAttention
// and inference kernels", GQA read amplification: one block per (sequence, KV
// head) computing all four query heads). Keys [s L, min((s+1) L, ctx)) arrive
// in 64-key tiles, one TMA box per 16-token page and half of the head
// dimension, found through the block table (same page, PagedAttention: token
// t in slot t % 16 of page table[t / 16]), into a ring of kStages tiles whose
// mbarriers count the bytes; m, l and the accumulator are carried across
// tiles. A segment writes its normalised output O_s = acc / l_s with (m_s, l_s).
//
// Merge kernel (same page, Flash-Decoding and the split-K merge exercise):
// m = max_s m_s, w_s = e^{m_s - m} l_s, O = sum_s w_s O_s / sum_s w_s, skipping
// segments with l_s = 0 (m_s = -inf). With one segment the split kernel writes
// the output directly and no partials are stored.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace attn {
namespace {

constexpr int kTile = 64;                      // keys per staged tile: four 16-token pages
constexpr int kPagesPerTile = kTile / ATTN_PAGE;
constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kStages = 2;                     // ring depth: one tile in flight while one is read (three blocks fit an SM)
constexpr int kHalfBytes = kTile * 128;        // 32 of the 64 dims of 64 rows, 128-byte swizzled
constexpr int kBoxBytes = ATTN_PAGE * 128;     // one page's rows of one d-half: a TMA box
constexpr int kStageBytes = 4 * kHalfBytes;    // K d-halves 0, 1, then V d-halves 0, 1 (32 KB)
constexpr int kPartFloats = kGroup * kD + 2 * kGroup;  // O_s for 4 heads, then m_s[4], l_s[4]
constexpr int kSkip = -2147483647 - 1;         // "no page": the tile's rows past the segment

// Shared memory: the ring (1024-byte aligned for the swizzle), then q [4][64],
// the tile's scores [4][64], its probabilities [64][4], alpha [4], the ring's
// barriers.
constexpr int kSmemQ = kStages * kStageBytes;
constexpr int kSmemSc = kSmemQ + kGroup * kD * 4;
constexpr int kSmemPk = kSmemSc + kGroup * kTile * 4;
constexpr int kSmemAl = kSmemPk + kTile * kGroup * 4;
constexpr int kSmemBar = kSmemAl + 16;
constexpr size_t kSplitSmem = kSmemBar + 8 * kStages + 1024;  // + slack for the alignment

// Byte offset of float f (0..31) of row r in a 128-byte-swizzled d-half: the
// 16-byte chunk c of row r sits at chunk c ^ (r mod 8) (the TMA swizzle).
__device__ __forceinline__ int swz(int r, int f) { return r * 128 + ((((f >> 2) ^ r) & 7) << 4) + (f & 3) * 4; }

struct DecodeArgs {
  const float* q;          // [B][32][64]
  const int* table;        // [B][max_blocks]
  const int* ctx_lens;     // [B]
  float* out;              // [B][32][64]
  float* parts;            // [B][8][splits][kPartFloats], or nullptr when splits == 1
  int B, max_blocks, num_pages, max_context, split_len, splits;
  unsigned* err;
  unsigned long long timeout_ns;  // a tile that has not landed by then is a fault
  int fault_skip_first;           // test hook: post the first tile's bytes, never load it
};

// mk, mv: the K and V page pools [num_pages * 16][8][64] as 2-D tensors
// (head * 64 + d, row), boxes of 32 floats x 16 rows, 128-byte swizzle.
__global__ void __launch_bounds__(kThreads)
decode_split_kernel(const __grid_constant__ CUtensorMap mk, const __grid_constant__ CUtensorMap mv, DecodeArgs a) {
  extern __shared__ __align__(16) uint8_t dsm_raw[];
  uint8_t* const dsm = dsm_raw + ((1024u - (tc::smem_u32(dsm_raw) & 1023u)) & 1023u);
  float (*qs)[kD] = reinterpret_cast<float (*)[kD]>(dsm + kSmemQ);
  // sc: the tile's scores [head][key]; pk: its probabilities [key][head]; al: alpha per head
  float (*sc)[kTile] = reinterpret_cast<float (*)[kTile]>(dsm + kSmemSc);
  float (*pk)[kGroup] = reinterpret_cast<float (*)[kGroup]>(dsm + kSmemPk);
  float* al = reinterpret_cast<float*>(dsm + kSmemAl);
  uint64_t* full = reinterpret_cast<uint64_t*>(dsm + kSmemBar);

  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int ctx = __ldg(a.ctx_lens + b);
  if (ctx < 0 || ctx > a.max_context || ctx > a.max_blocks * 16) {
    record_error(a.err, kDevErrBounds);
    ctx = ctx < 0 ? 0 : min(a.max_context, a.max_blocks * 16);
  }
  const int k0 = s * a.split_len;
  const int k1 = min(k0 + a.split_len, ctx);
  float* part = a.parts ? a.parts + (((size_t)b * kHKV + g) * a.splits + s) * kPartFloats : nullptr;

  if (k0 >= k1) {  // empty segment (or an empty sequence): weight zero in the merge
    if (part && tid < kGroup) {
      part[kGroup * kD + tid] = -INFINITY;
      part[kGroup * kD + kGroup + tid] = 0.f;
    }
    if (!part) {  // single segment and ctx == 0: no key to attend to
      for (int i = tid; i < kGroup * kD; i += kThreads)
        a.out[((size_t)b * kHQ + g * kGroup) * kD + i] = 0.f;
    }
    return;
  }

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) tc::mbar_init(&full[i], 1);
    tc::fence_mbar_init();
  }
  for (int i = tid; i < kGroup * kD; i += kThreads)
    qs[i / kD][i % kD] = a.q[((size_t)b * kHQ + g * kGroup) * kD + i];
  __syncthreads();

  const int ntiles = (k1 - k0 + kTile - 1) / kTile;
  const int* trow = a.table + (size_t)b * a.max_blocks;
  // Warp 0, lane i < 4: the physical page of the i-th page of tile n, or kSkip
  // when it starts at or past the segment's end (t < k1 <= ctx keeps the table
  // index below max_blocks).
  auto page_of = [&](int n) -> int {
    const int t = k0 + n * kTile + lane * ATTN_PAGE;
    if (lane >= kPagesPerTile || n >= ntiles || t >= k1) return kSkip;
    return __ldg(trow + (t >> 4));
  };
  // Warp 0 fills tile n's stage: lane 0 posts the bytes of the pages present,
  // then lane i loads page i's rows of both d-halves of K and of V (four boxes).
  // A table entry outside [0, num_pages) is recorded and loaded from past the
  // pool's end, which TMA fills with zeros.
  auto issue = [&](int n, int pg) {
    const int st = n % kStages;
    uint8_t* stage = dsm + st * kStageBytes;
    const bool has = pg != kSkip;
    const unsigned npg = __popc(__ballot_sync(0xffffffffu, has));
    if (lane == 0) tc::mbar_arrive_expect_tx(&full[st], npg * 4u * kBoxBytes);
    __syncwarp();
    if (has && !(a.fault_skip_first && n == 0)) {
      int y = pg;
      if (pg < 0 || pg >= a.num_pages) {
        record_error(a.err, kDevErrBounds);
        y = a.num_pages;
      }
      y *= ATTN_PAGE;
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        tc::tma_load_2d(stage + q4 * kHalfBytes + lane * kBoxBytes, q4 < 2 ? &mk : &mv, &full[st],
                        g * kD + (q4 & 1) * 32, y);
    }
  };

  // Scores and the online update: warp h is query head h and lane l scores
  // keys l and l + 32 of the tile, so the scores stay in registers.
  // Weighted sum: warp w takes keys 16 w .. 16 w + 15 of every tile for all four
  // heads, lane = head dims 2 lane, 2 lane + 1; the four warps' sums share each
  // head's reference maximum and are added at the end.
  float m = -INFINITY, l = 0.f;
  float o[kGroup][2];
#pragma unroll
  for (int h = 0; h < kGroup; ++h) o[h][0] = o[h][1] = 0.f;

  int pg_next = kSkip;
  if (warp == 0) {
    for (int n = 0; n < kStages - 1 && n < ntiles; ++n) issue(n, page_of(n));
    pg_next = page_of(kStages - 1);
  }
  int it = 0;
  bool failed = false;
  for (; it < ntiles; ++it) {
    const int st = it % kStages;
    const int t0 = k0 + it * kTile;
    // The stage of tile it + kStages - 1 held tile it - 1, which every thread
    // finished with before the previous iteration's last barrier.
    if (warp == 0 && it + kStages - 1 < ntiles) {
      issue(it + kStages - 1, pg_next);
      pg_next = page_of(it + kStages);  // its latency is spent on this tile's work
    }
    const bool ok = tc::mbar_wait(&full[st], (it / kStages) & 1, a.timeout_ns);
    const uint8_t* kt = dsm + st * kStageBytes;
    const uint8_t* vt = kt + 2 * kHalfBytes;

    // Scores of keys `lane` and `lane + 32` against head `warp`, scale 1/8,
    // then the head's tile maximum, alpha and probabilities. Keys past the
    // segment read whatever the page slot holds (NaN included) and get score
    // -inf. (After an expired wait the values are garbage; nothing is stored
    // from them.)
    {
      float d0 = 0.f, d1 = 0.f;
#pragma unroll
      for (int d4 = 0; d4 < kD / 4; ++d4) {
        const float4 qa = *reinterpret_cast<const float4*>(&qs[warp][d4 * 4]);
        const uint8_t* kh = kt + (d4 >> 3) * kHalfBytes;
        const float4 ka = *reinterpret_cast<const float4*>(kh + swz(lane, (d4 & 7) * 4));
        const float4 kb = *reinterpret_cast<const float4*>(kh + swz(lane + 32, (d4 & 7) * 4));
        d0 = fmaf(qa.x, ka.x, fmaf(qa.y, ka.y, fmaf(qa.z, ka.z, fmaf(qa.w, ka.w, d0))));
        d1 = fmaf(qa.x, kb.x, fmaf(qa.y, kb.y, fmaf(qa.z, kb.z, fmaf(qa.w, kb.w, d1))));
      }
      const float s0 = t0 + lane < k1 ? d0 * kScale : -INFINITY;
      const float s1 = t0 + lane + 32 < k1 ? d1 * kScale : -INFINITY;
      float mx = fmaxf(s0, s1);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float mnew = fmaxf(m, mx);  // finite: the tile holds at least one valid key
      const float alpha = exp2f((m - mnew) * kLog2e);  // 0 while m = -inf
      const float p0 = exp2f((s0 - mnew) * kLog2e), p1 = exp2f((s1 - mnew) * kLog2e);
      float ps = p0 + p1;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
      l = fmaf(l, alpha, ps);
      m = mnew;
      pk[lane][warp] = p0;
      pk[lane + 32][warp] = p1;
      if (lane == 0) al[warp] = alpha;
    }
    // Every thread's wait either succeeded or it gives up with the others.
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }

    // O_w += P V over this warp's 16 keys, all four heads. A key past the
    // segment is skipped, not weighted by zero: its slot may hold NaN.
    {
      const float4 a4 = *reinterpret_cast<const float4*>(al);
      o[0][0] *= a4.x; o[0][1] *= a4.x;
      o[1][0] *= a4.y; o[1][1] *= a4.y;
      o[2][0] *= a4.z; o[2][1] *= a4.z;
      o[3][0] *= a4.w; o[3][1] *= a4.w;
      const uint8_t* vb = vt + (lane >> 4) * kHalfBytes;
      const int f = (2 * lane) & 31;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int key = 16 * warp + j;
        if (t0 + key >= k1) break;
        const float4 p4 = *reinterpret_cast<const float4*>(&pk[key][0]);
        const float2 vv = *reinterpret_cast<const float2*>(vb + swz(key, f));
        o[0][0] = fmaf(p4.x, vv.x, o[0][0]);
        o[0][1] = fmaf(p4.x, vv.y, o[0][1]);
        o[1][0] = fmaf(p4.y, vv.x, o[1][0]);
        o[1][1] = fmaf(p4.y, vv.y, o[1][1]);
        o[2][0] = fmaf(p4.z, vv.x, o[2][0]);
        o[2][1] = fmaf(p4.z, vv.y, o[2][1]);
        o[3][0] = fmaf(p4.w, vv.x, o[3][0]);
        o[3][1] = fmaf(p4.w, vv.y, o[3][1]);
      }
    }
    __syncthreads();  // before tile it + kStages refills this stage and sc, pk, al are rewritten
  }

  if (failed) {
    // A tile did not land in time: record it and give the copies still in
    // flight (tiles it .. it + kStages - 1: the last was issued before the
    // wait) a bounded wait before the block's shared memory is released. The
    // output is not written. The segment's partial record is written empty
    // (m = -inf, l = 0), as for an empty segment, so the merge never weights
    // whatever an earlier call left in a reused workspace or scratch.
    if (part && tid < kGroup) {
      part[kGroup * kD + tid] = -INFINITY;
      part[kGroup * kD + kGroup + tid] = 0.f;
    }
    if (tid == 0) {
      record_error(a.err, kDevErrTimeout);
      const int last = min(ntiles - 1, it + kStages - 1);
      for (int n = it; n <= last; ++n) tc::mbar_wait(&full[n % kStages], (n / kStages) & 1, a.timeout_ns);
    }
    return;
  }

  // Sum the four warps' accumulators (stage 0 is free: every tile issued has
  // been waited for), then one division per element by the head's l.
  float* acc = reinterpret_cast<float*>(dsm);  // [4 warps][4 heads][64]
#pragma unroll
  for (int h = 0; h < kGroup; ++h)
    *reinterpret_cast<float2*>(acc + (warp * kGroup + h) * kD + 2 * lane) = make_float2(o[h][0], o[h][1]);
  if (lane == 0) {
    al[warp] = l;  // head `warp`'s l (al is no longer needed)
    sc[0][warp] = m;
  }
  __syncthreads();
  {
    const int h = tid >> 5, dl = tid & 31;  // thread = (head, pair of head dims)
    float O0 = 0.f, O1 = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float2 x = *reinterpret_cast<const float2*>(acc + (w * kGroup + h) * kD + 2 * dl);
      O0 += x.x;
      O1 += x.y;
    }
    const float lh = al[h], mh = sc[0][h];
    if (!part) {
      *reinterpret_cast<float2*>(a.out + ((size_t)b * kHQ + g * kGroup + h) * kD + 2 * dl) =
          make_float2(O0 / lh, O1 / lh);
    } else {
      *reinterpret_cast<float2*>(part + h * kD + 2 * dl) = make_float2(O0 / lh, O1 / lh);
      if (dl == 0) {
        part[kGroup * kD + h] = mh;
        part[kGroup * kD + kGroup + h] = lh;
      }
    }
  }
  // This block's partial is written: the merge grid may be scheduled (it
  // still waits for this whole grid to finish before reading any partial).
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// One block per (sequence, query head); thread d owns head dimension d.
__global__ void __launch_bounds__(kD)
decode_merge_kernel(DecodeArgs a) {
  // Launched as a programmatic dependent of the split kernel: wait until that
  // grid has completed and its partials are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.x, h = blockIdx.y, d = threadIdx.x;
  const int g = h / kGroup, hl = h % kGroup;
  const float* base = a.parts + ((size_t)b * kHKV + g) * a.splits * kPartFloats;
  float m = -INFINITY;
  for (int s = 0; s < a.splits; ++s) {
    const float* part = base + (size_t)s * kPartFloats;
    if (part[kGroup * kD + kGroup + hl] > 0.f) m = fmaxf(m, part[kGroup * kD + hl]);
  }
  float num = 0.f, den = 0.f;
  for (int s = 0; s < a.splits; ++s) {
    const float* part = base + (size_t)s * kPartFloats;
    const float ls = part[kGroup * kD + kGroup + hl];
    if (!(ls > 0.f)) continue;  // an empty segment has no weight (and m_s = -inf)
    const float w = exp2f((part[kGroup * kD + hl] - m) * kLog2e) * ls;
    num = fmaf(w, part[hl * kD + d], num);
    den += w;
  }
  a.out[((size_t)b * kHQ + h) * kD + d] = den > 0.f ? num / den : 0.f;
}

}  // namespace

// The library's own partials buffer for attn_decode_paged_noalloc: a fixed
// array in device global memory, created with the module, so that entry point
// needs neither a workspace from the caller nor an allocation of its own. Every
// call on a device shares it. Nothing in it has to start at zero: the split
// kernel writes each (sequence, KV head, segment) record, m_s and l_s always
// and O_s whenever l_s > 0, before the merge kernel of the same call reads it.
static __device__ __align__(256) float g_decode_scratch[kDecodeScratchBytes / sizeof(float)];

cudaError_t decode_scratch(float** ptr) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static float* addr[kMaxDev] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {  // once per device, with that device current
    void* a = nullptr;
    e = cudaGetSymbolAddress(&a, g_decode_scratch);
    if (e != cudaSuccess) return e;
    addr[dev] = static_cast<float*>(a);
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

namespace {

// Per device: the shared-memory opt-in and how many split blocks fit at once.
struct DecodeDevice {
  bool ready = false;
  int slots = 0;  // resident split blocks on the whole device
};

int decode_device(DecodeDevice** out) {
  constexpr int kMaxDev = 64;
  static std::mutex mu;
  static DecodeDevice devs[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return ATTN_ECUDA;
  std::lock_guard<std::mutex> lock(mu);
  DecodeDevice& d = devs[dev];
  if (!d.ready) {
    int sms = 0, per_sm = 0;
    if (cudaFuncSetAttribute(decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSplitSmem) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_split_kernel, kThreads, kSplitSmem) !=
            cudaSuccess)
      return ATTN_ECUDA;
    d.slots = sms * (per_sm > 0 ? per_sm : 1);
    d.ready = true;
  }
  *out = &d;
  return ATTN_OK;
}

// The driver's tensor-map encoder, looked up once (a function-local static is
// initialised once even when the first calls come from several threads).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// A page pool [num_pages * 16][8][64] fp32 as the 2-D tensor (head * 64 + d,
// row); a box is 32 floats (one 128-byte swizzle row) x the 16 rows of a page.
int encode_page_pool(const float* base, int num_pages, CUtensorMap* map) {
  auto enc = tensor_map_encoder();
  if (!enc) return ATTN_ETMA;
  const cuuint32_t ones[2] = {1, 1};
  const cuuint64_t dims[2] = {(cuuint64_t)kHKV * kD, (cuuint64_t)num_pages * ATTN_PAGE};
  const cuuint64_t strides[1] = {(cuuint64_t)kHKV * kD * 4};
  const cuuint32_t box[2] = {32, ATTN_PAGE};
  if (enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box, ones,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return ATTN_ETMA;
  return ATTN_OK;
}

}  // namespace

int decode_slots(int* slots) {
  DecodeDevice* d = nullptr;
  const int rc = decode_device(&d);
  if (rc == ATTN_OK) *slots = d->slots;
  return rc;
}

int decode_splits(int B, int max_context, int splits_hint, int slots, int* split_len) {
  int splits = splits_hint;
  if (splits <= 0) {
    // Segments of at least 256 keys, as many as fill the resident blocks
    // best: blocks / (waves x slots), less 0.04 for each extra wave.
    const long long pairs = (long long)B * kHKV;
    const int most = (max_context + 255) / 256;
    const int top = most < 64 ? most : 64;
    double best_score = -1.0;
    splits = 1;
    for (int s = 1; s <= top && slots > 0 && pairs > 0; ++s) {
      const long long blocks = pairs * s;
      const long long waves = (blocks + slots - 1) / slots;
      const double score = (double)blocks / (double)(waves * slots) - 0.04 * (double)(waves - 1);
      if (score > best_score + 1e-9) {
        best_score = score;
        splits = s;
      }
    }
  }
  if (splits < 1) splits = 1;
  const int per = (max_context + splits - 1) / splits;
  *split_len = ((per + kTile - 1) / kTile) * kTile;
  if (*split_len < kTile) *split_len = kTile;
  return (max_context + *split_len - 1) / *split_len > 0 ? (max_context + *split_len - 1) / *split_len : 1;
}

size_t decode_workspace_bytes(int B, int splits) {
  return splits <= 1 ? 0 : (size_t)B * kHKV * splits * kPartFloats * sizeof(float);
}

int launch_decode(const float* q, const float* k_pages, const float* v_pages, const int* table,
                  const int* ctx_lens, float* out, float* parts, int B, int max_blocks, int num_pages,
                  int max_context, int split_len, int splits, unsigned* err, cudaStream_t stream, int fault) {
  DecodeDevice* d = nullptr;
  int rc = decode_device(&d);
  if (rc != ATTN_OK) return rc;
  alignas(64) CUtensorMap mk, mv;
  if ((rc = encode_page_pool(k_pages, num_pages, &mk)) != ATTN_OK ||
      (rc = encode_page_pool(v_pages, num_pages, &mv)) != ATTN_OK)
    return rc;
  DecodeArgs a{q, table, ctx_lens, out, splits > 1 ? parts : nullptr,
               B, max_blocks, num_pages, max_context, split_len, splits, err,
               fault ? 20000000ull : 2000000000ull, fault};
  decode_split_kernel<<<dim3(splits, kHKV, B), kThreads, kSplitSmem, stream>>>(mk, mv, a);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ELAUNCH;
  if (splits > 1) {
    // The merge starts as soon as every split block has written its partial
    // (programmatic dependent launch) instead of after the split grid drains.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(B, kHQ);
    cfg.blockDim = dim3(kD);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_merge_kernel, a) != cudaSuccess) return ATTN_ELAUNCH;
  }
  return ATTN_OK;
}

}  // namespace attn
