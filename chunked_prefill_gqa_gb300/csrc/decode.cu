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
// in 64-key tiles through a two-stage cp.async ring, each row found through
// the block table (same page, PagedAttention: token t in slot t % 16 of page
// table[t / 16]); m, l and the accumulator are carried across tiles. A segment
// writes its normalised output O_s = acc / l_s with (m_s, l_s).
//
// Merge kernel (same page, Flash-Decoding and the split-K merge exercise):
// m = max_s m_s, w_s = e^{m_s - m} l_s, O = sum_s w_s O_s / sum_s w_s, skipping
// segments with l_s = 0 (m_s = -inf). With one segment the split kernel writes
// the output directly and no partials are stored.
#include <mutex>

#include "common.cuh"

namespace attn {
namespace {

constexpr int kTile = 64;            // keys per staged tile
constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kLdK = 68;             // padded K row (floats): 16-byte loads of 8 consecutive keys hit 8 bank groups
constexpr int kPartFloats = kGroup * kD + 2 * kGroup;  // O_s for 4 heads, then m_s[4], l_s[4]
constexpr size_t kSplitSmem =
    sizeof(float) * (2 * kTile * kLdK + 2 * kTile * kD + kGroup * kD + 2 * kGroup * kTile + kGroup);  // 70,672 B

__device__ __forceinline__ void cp_async16(float* dst, const float* src, bool valid) {
  const unsigned s = (unsigned)__cvta_generic_to_shared(dst);
  const int n = valid ? 16 : 0;  // n == 0 writes zeros and reads nothing
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(s), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

struct DecodeArgs {
  const float* q;          // [B][32][64]
  const float* k_pages;    // [num_pages][16][8][64]
  const float* v_pages;
  const int* table;        // [B][max_blocks]
  const int* ctx_lens;     // [B]
  float* out;              // [B][32][64]
  float* parts;            // [B][8][splits][kPartFloats], or nullptr when splits == 1
  int B, max_blocks, num_pages, max_context, split_len, splits;
  unsigned* err;
};

// Stage keys [k0, k0 + 64) of KV head g of sequence b (rows at or past `end`
// become zeros; a table entry outside [0, num_pages) is recorded and read as
// zeros).
__device__ __forceinline__ void load_tile(const DecodeArgs& a, int b, int g, int k0, int end, float* ks,
                                          float* vs, int tid) {
#pragma unroll
  for (int it = 0; it < (kTile * kD / 4) / kThreads; ++it) {
    const int idx = tid + it * kThreads;
    const int key = idx >> 4, c4 = idx & 15;
    const int t = k0 + key;
    bool valid = t < end;
    size_t row = 0;
    if (valid) {
      const int page = __ldg(a.table + (size_t)b * a.max_blocks + (t >> 4));
      if (page < 0 || page >= a.num_pages) {
        record_error(a.err, kDevErrBounds);
        valid = false;
      } else {
        row = (size_t)page * 16 + (t & 15);
      }
    }
    const size_t src = (row * kHKV + g) * kD + c4 * 4;
    cp_async16(ks + key * kLdK + c4 * 4, a.k_pages + src, valid);
    cp_async16(vs + key * kD + c4 * 4, a.v_pages + src, valid);
  }
}

__global__ void __launch_bounds__(kThreads)
decode_split_kernel(DecodeArgs a) {
  extern __shared__ __align__(16) float dsm[];
  float* const ks0 = dsm;                         // two K tiles, padded rows
  float* const vs0 = dsm + 2 * kTile * kLdK;       // two V tiles
  float (*qs)[kD] = reinterpret_cast<float (*)[kD]>(dsm + 2 * kTile * kLdK + 2 * kTile * kD);
  float (*sc)[kTile] = reinterpret_cast<float (*)[kTile]>(dsm + 2 * kTile * kLdK + 2 * kTile * kD + kGroup * kD);
  // sc: the tile's scores [head][key]; pk: its probabilities [key][head]; al: alpha per head
  float (*pk)[kGroup] = reinterpret_cast<float (*)[kGroup]>(&sc[0][0] + kGroup * kTile);
  float* al = &pk[0][0] + kTile * kGroup;

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

  for (int i = tid; i < kGroup * kD; i += kThreads)
    qs[i / kD][i % kD] = a.q[((size_t)b * kHQ + g * kGroup) * kD + i];

  // Score layout: thread (key = tid % 64, head pair = tid / 64).
  const int skey = tid & 63, hp = (tid >> 6) * 2;
  // Softmax: warp = head (m and l live in warp `warp`'s registers for head `warp`).
  // Weighted sum: warp w takes keys 16 w .. 16 w + 15 of every tile for all four
  // heads, lane = head dims 2 lane, 2 lane + 1; the four warps' sums share each
  // head's reference maximum and are added at the end.
  float m = -INFINITY, l = 0.f;
  float o[kGroup][2];
#pragma unroll
  for (int h = 0; h < kGroup; ++h) o[h][0] = o[h][1] = 0.f;

  const int ntiles = (k1 - k0 + kTile - 1) / kTile;
  load_tile(a, b, g, k0, k1, ks0, vs0, tid);
  cp_async_commit();
  for (int it = 0; it < ntiles; ++it) {
    const int buf = it & 1;
    const int t0 = k0 + it * kTile;
    if (it + 1 < ntiles) {
      load_tile(a, b, g, t0 + kTile, k1, ks0 + (buf ^ 1) * kTile * kLdK, vs0 + (buf ^ 1) * kTile * kD, tid);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();

    // Scores of this thread's key against two query heads, scale 1/8.
    {
      const float* kr = ks0 + buf * kTile * kLdK + skey * kLdK;
      float d0 = 0.f, d1 = 0.f;
#pragma unroll
      for (int d4 = 0; d4 < kD / 4; ++d4) {
        const float4 kv = *reinterpret_cast<const float4*>(kr + d4 * 4);
        const float4 qa = *reinterpret_cast<const float4*>(&qs[hp][d4 * 4]);
        const float4 qb = *reinterpret_cast<const float4*>(&qs[hp + 1][d4 * 4]);
        d0 = fmaf(qa.x, kv.x, fmaf(qa.y, kv.y, fmaf(qa.z, kv.z, fmaf(qa.w, kv.w, d0))));
        d1 = fmaf(qb.x, kv.x, fmaf(qb.y, kv.y, fmaf(qb.z, kv.z, fmaf(qb.w, kv.w, d1))));
      }
      const bool valid = t0 + skey < k1;
      sc[hp][skey] = valid ? d0 * kScale : -INFINITY;
      sc[hp + 1][skey] = valid ? d1 * kScale : -INFINITY;
    }
    __syncthreads();

    // Online update for head `warp`: tile max, alpha, probabilities.
    {
      const int h = warp;
      const float s0 = sc[h][lane], s1 = sc[h][lane + 32];
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
      pk[lane][h] = p0;
      pk[lane + 32][h] = p1;
      if (lane == 0) al[h] = alpha;
    }
    __syncthreads();

    // O_w += P V over this warp's 16 keys, all four heads.
    {
      const float4 a4 = *reinterpret_cast<const float4*>(al);
      o[0][0] *= a4.x; o[0][1] *= a4.x;
      o[1][0] *= a4.y; o[1][1] *= a4.y;
      o[2][0] *= a4.z; o[2][1] *= a4.z;
      o[3][0] *= a4.w; o[3][1] *= a4.w;
      const float* vb = vs0 + buf * kTile * kD + (16 * warp) * kD + 2 * lane;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float4 p4 = *reinterpret_cast<const float4*>(&pk[16 * warp + j][0]);
        const float2 vv = *reinterpret_cast<const float2*>(vb + j * kD);
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
    __syncthreads();  // before the next tile overwrites sc, pk, al, ks, vs
  }

  // Sum the four warps' accumulators (the first K tile buffer is free now),
  // then one division per element by the head's l.
  float* acc = ks0;  // [4 warps][4 heads][64]
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
}

// One block per (sequence, query head); thread d owns head dimension d.
__global__ void __launch_bounds__(kD)
decode_merge_kernel(DecodeArgs a) {
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

int decode_splits(int B, int max_context, int splits_hint, int num_sms, int* split_len) {
  int splits = splits_hint;
  if (splits <= 0) {
    // Enough blocks for two waves of the SMs, segments of at least 256 keys.
    const int want = (2 * num_sms + B * kHKV - 1) / (B * kHKV);
    const int most = (max_context + 255) / 256;
    splits = want < most ? want : most;
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

cudaError_t launch_decode(const float* q, const float* k_pages, const float* v_pages, const int* table,
                          const int* ctx_lens, float* out, float* parts, int B, int max_blocks, int num_pages,
                          int max_context, int split_len, int splits, unsigned* err, cudaStream_t stream) {
  static bool configured[64] = {};  // the shared-memory opt-in is per device
  static std::mutex mu;
  int dev = 0;
  cudaError_t e0 = cudaGetDevice(&dev);
  if (e0 != cudaSuccess) return e0;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!configured[dev]) {
    e0 = cudaFuncSetAttribute(decode_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSplitSmem);
    if (e0 != cudaSuccess) return e0;
    configured[dev] = true;
  }
  DecodeArgs a{q, k_pages, v_pages, table, ctx_lens, out, splits > 1 ? parts : nullptr,
               B, max_blocks, num_pages, max_context, split_len, splits, err};
  decode_split_kernel<<<dim3(splits, kHKV, B), kThreads, kSplitSmem, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || splits <= 1) return e;
  decode_merge_kernel<<<dim3(B, kHQ), kD, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace attn
