// api.cu -- the extern "C" entry points of libattnprefill.so: argument
// validation, the device check, the device error word and dispatch to the
// kernel launchers. No entry point allocates device memory.
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "common.cuh"

namespace attn {
namespace {

// The device error word: kernels record the first internal fault here
// (a bounded wait that expired, a failed bounds check) instead of trapping.
__device__ unsigned g_error_word;

constexpr int kMaxDevices = 64;

struct DeviceState {
  bool checked = false;
  bool supported = false;
  unsigned* err = nullptr;  // device address of g_error_word on this device
};
DeviceState g_devices[kMaxDevices];
std::mutex g_devices_mu;  // first use of a device may come from several host threads

// Looks up (once per device) whether the current device is sm_103 and where
// its error word lives. Returns an ATTN_* code.
int current_device(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ECUDA;
  std::lock_guard<std::mutex> lock(g_devices_mu);
  DeviceState& st = g_devices[dev];
  if (!st.checked) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return ATTN_ECUDA;
    st.supported = (major == 10 && minor == 3);
    if (st.supported) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_error_word) != cudaSuccess) return ATTN_ECUDA;
      st.err = static_cast<unsigned*>(addr);
    }
    st.checked = true;
  }
  if (!st.supported) return ATTN_EDEVICE;
  *out = &st;
  return ATTN_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// Shared validation of every compute entry point. On success fills `p`.
int prepare(const float* q, const float* k, const float* v, float* out, int C, int P,
            Problem* p) {
  if (C < 0 || P < 0) return ATTN_EINVAL;
  if (C > ATTN_MAX_TOKENS || (long long)P + C > ATTN_MAX_TOKENS) return ATTN_ERANGE;
  if (C == 0) return ATTN_OK;  // empty chunk: nothing to do, pointers unused
  if (!q || !k || !v || !out) return ATTN_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return ATTN_EALIGN;
  DeviceState* st = nullptr;
  const int rc = current_device(&st);
  if (rc != ATTN_OK) return rc;
  *p = Problem{q, k, v, out, C, P, st->err};
  return ATTN_OK;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ELAUNCH; }

int sm_count(int* n) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ECUDA;
  if (cudaDeviceGetAttribute(n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return ATTN_ECUDA;
  return ATTN_OK;
}

// Shape checks shared by the decode entry points.
int decode_shape_ok(int B, int maxBlocks, int numPages, int maxContext, int numSplits) {
  if (B < 0 || maxBlocks < 1 || numPages < 1 || maxContext < 0 || numSplits < 0) return ATTN_EINVAL;
  if (B > 65535 || (long long)maxBlocks * ATTN_PAGE > ATTN_MAX_TOKENS || numPages > ATTN_MAX_TOKENS / ATTN_PAGE ||
      maxContext > maxBlocks * ATTN_PAGE)
    return ATTN_ERANGE;
  return ATTN_OK;
}

// Shared validation of the score-matrix entry points: sizes, and (for C > 0)
// the device. The pointers are checked by each caller.
int naive_prepare(int C, int P, DeviceState** st) {
  if (C < 0 || P < 0) return ATTN_EINVAL;
  if (C > ATTN_MAX_TOKENS || (long long)P + C > ATTN_MAX_TOKENS || C > naive_max_rows()) return ATTN_ERANGE;
  if (C == 0) return ATTN_OK;
  return current_device(st);
}

// ---------------------------------------------------------------------------
// Host-buffer calls: the chunk is run as up to kMaxSlices consecutive
// sub-chunks of whole 32-row query tiles, each one full round of units.
// Sub-chunk s (rows r0 .. r1-1) is the prefill of those rows against positions
// 0 .. P+r1-1, the same rows of the whole call's result. Its copy-in adds only
// its query rows and the K/V rows past the previous sub-chunk's end, so
// copy-in of s+1 and copy-out of s-1 overlap the compute of s; sub-chunks
// compute alternately on the caller's stream and a library stream, so the
// next one's blocks take SMs as the previous one's leave.
constexpr int kMaxSlices = 4;

struct HostPipe {
  std::mutex mu;  // held for a whole enqueue: every call re-records the events
  bool made = false;
  int sms = 0;
  cudaStream_t in = nullptr, out = nullptr, comp2 = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t loaded[kMaxSlices] = {}, computed[kMaxSlices] = {};
};
HostPipe g_pipes[kMaxDevices];

// Slice boundaries: each slice is one full round of units, sms / 8 query
// tiles (8 KV heads per tile: one unit per SM), the last one the remainder; with
// more than kMaxSlices such rounds, kMaxSlices equal slices instead.
int plan_slices(int C, int sms, int bounds[kMaxSlices + 1]) {
  const int tiles = (C + 31) / 32;
  int per = sms / ATTN_HKV;
  if (per < 1) per = 1;
  int n = (tiles + per - 1) / per;
  if (n > kMaxSlices) {
    n = kMaxSlices;
    per = (tiles + n - 1) / n;
  }
  bounds[0] = 0;
  for (int s = 0; s < n; ++s) {
    const long long end = (long long)((s + 1) * per < tiles ? (s + 1) * per : tiles) * 32;
    bounds[s + 1] = end < C ? (int)end : C;
  }
  return n;
}

// The current device's pipe, its streams and events made on first use.
// Called with pipe->mu held.
int make_pipe(HostPipe* hp) {
  if (hp->made) return ATTN_OK;
  if (cudaStreamCreateWithFlags(&hp->in, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&hp->out, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&hp->comp2, cudaStreamNonBlocking) != cudaSuccess ||
      cudaEventCreateWithFlags(&hp->start, cudaEventDisableTiming) != cudaSuccess ||
      cudaEventCreateWithFlags(&hp->done, cudaEventDisableTiming) != cudaSuccess)
    return ATTN_ECUDA;
  for (int s = 0; s < kMaxSlices; ++s)
    if (cudaEventCreateWithFlags(&hp->loaded[s], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp->computed[s], cudaEventDisableTiming) != cudaSuccess)
      return ATTN_ECUDA;
  if (sm_count(&hp->sms) != ATTN_OK) return ATTN_ECUDA;
  hp->made = true;
  return ATTN_OK;
}

using Launcher = int (*)(const Problem&, cudaStream_t);

// kv_row: bytes of one position of kCache (and vCache), 8 heads x 64 values.
int run_from_host(const float* q_h, const void* k_h, const void* v_h, float* out_h, float* q_d, void* k_d,
                  void* v_d, float* out_d, size_t kv_row, int C, int P, cudaStream_t stream, Launcher launch) {
  if (C > 0 && (!q_h || !k_h || !v_h || !out_h)) return ATTN_EINVAL;
  Problem p{};
  int rc = prepare(q_d, static_cast<const float*>(k_d), static_cast<const float*>(v_d), out_d, C, P, &p);
  if (rc != ATTN_OK || C == 0) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ECUDA;
  HostPipe* hp = &g_pipes[dev];  // dev < kMaxDevices: prepare checked it
  std::lock_guard<std::mutex> lock(hp->mu);
  rc = make_pipe(hp);
  if (rc != ATTN_OK) return rc;
  if (cudaEventRecord(hp->start, stream) != cudaSuccess || cudaStreamWaitEvent(hp->in, hp->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(hp->out, hp->start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(hp->comp2, hp->start, 0) != cudaSuccess)
    return ATTN_ECUDA;
  constexpr size_t kQRow = sizeof(float) * ATTN_HQ * ATTN_D;
  auto* kd = static_cast<char*>(k_d);
  auto* vd = static_cast<char*>(v_d);
  const auto* kh = static_cast<const char*>(k_h);
  const auto* vh = static_cast<const char*>(v_h);
  int bounds[kMaxSlices + 1];
  const int n = plan_slices(C, hp->sms, bounds);
  size_t kv0 = 0;
  for (int s = 0; s < n && rc == ATTN_OK; ++s) {
    const int r0 = bounds[s], r1 = bounds[s + 1];
    const size_t q0 = (size_t)r0 * kQRow, nq = (size_t)(r1 - r0) * kQRow;
    const size_t kv1 = ((size_t)P + r1) * kv_row;
    if (cudaMemcpyAsync((char*)q_d + q0, (const char*)q_h + q0, nq, cudaMemcpyDefault, hp->in) != cudaSuccess ||
        cudaMemcpyAsync(kd + kv0, kh + kv0, kv1 - kv0, cudaMemcpyDefault, hp->in) != cudaSuccess ||
        cudaMemcpyAsync(vd + kv0, vh + kv0, kv1 - kv0, cudaMemcpyDefault, hp->in) != cudaSuccess ||
        cudaEventRecord(hp->loaded[s], hp->in) != cudaSuccess ||
        cudaStreamWaitEvent((s & 1) ? hp->comp2 : stream, hp->loaded[s], 0) != cudaSuccess) {
      rc = ATTN_ECUDA;
      break;
    }
    kv0 = kv1;
    Problem ps = p;
    ps.q = q_d + (size_t)r0 * ATTN_HQ * ATTN_D;
    ps.out = out_d + (size_t)r0 * ATTN_HQ * ATTN_D;
    ps.C = r1 - r0;
    ps.P = P + r0;
    // Consecutive sub-chunks alternate between two streams, so the next one's
    // blocks take SMs as the previous one's finish.
    cudaStream_t cs = (s & 1) ? hp->comp2 : stream;
    rc = launch(ps, cs);
    if (rc != ATTN_OK) break;
    if (cudaEventRecord(hp->computed[s], cs) != cudaSuccess ||
        cudaStreamWaitEvent(hp->out, hp->computed[s], 0) != cudaSuccess ||
        cudaMemcpyAsync((char*)out_h + q0, (const char*)out_d + q0, nq, cudaMemcpyDefault, hp->out) != cudaSuccess)
      rc = ATTN_ECUDA;
  }
  // Whatever was enqueued, `stream` waits for both library streams.
  const bool joined = cudaEventRecord(hp->done, hp->in) == cudaSuccess &&
                      cudaStreamWaitEvent(stream, hp->done, 0) == cudaSuccess &&
                      cudaEventRecord(hp->done, hp->comp2) == cudaSuccess &&
                      cudaStreamWaitEvent(stream, hp->done, 0) == cudaSuccess &&
                      cudaEventRecord(hp->done, hp->out) == cudaSuccess &&
                      cudaStreamWaitEvent(stream, hp->done, 0) == cudaSuccess;
  if (rc == ATTN_OK && !joined) rc = ATTN_ECUDA;
  return rc;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" int attn_prefill_host(const float* q_host, const float* kCache_host, const float* vCache_host,
                                 float* out_host, float* q_dev, float* kCache_dev, float* vCache_dev,
                                 float* out_dev, int C, int P, cudaStream_t stream) {
  return run_from_host(q_host, kCache_host, vCache_host, out_host, q_dev, kCache_dev, vCache_dev, out_dev,
                       sizeof(float) * ATTN_HKV * ATTN_D, C, P, stream, launch_tc);
}

extern "C" int attn_prefill_bf16x3_host(const float* q_host, const float* kCache_host, const float* vCache_host,
                                        float* out_host, float* q_dev, float* kCache_dev, float* vCache_dev,
                                        float* out_dev, int C, int P, cudaStream_t stream) {
  return run_from_host(q_host, kCache_host, vCache_host, out_host, q_dev, kCache_dev, vCache_dev, out_dev,
                       sizeof(float) * ATTN_HKV * ATTN_D, C, P, stream, launch_tc_bf16x3);
}

extern "C" int attn_prefill_bf16kv_host(const float* q_host, const uint16_t* kCache_host,
                                        const uint16_t* vCache_host, float* out_host, float* q_dev,
                                        uint16_t* kCache_dev, uint16_t* vCache_dev, float* out_dev, int C, int P,
                                        cudaStream_t stream) {
  return run_from_host(q_host, kCache_host, vCache_host, out_host, q_dev, kCache_dev, vCache_dev, out_dev,
                       sizeof(uint16_t) * ATTN_HKV * ATTN_D, C, P, stream, launch_tc_bf16);
}

extern "C" int attn_prefill(const float* q, const float* kCache, const float* vCache, float* out,
                            int C, int P, cudaStream_t stream) {
  Problem p{};
  const int rc = prepare(q, kCache, vCache, out, C, P, &p);
  if (rc != ATTN_OK || C == 0) return rc;
  return launch_tc(p, stream);
}

extern "C" int attn_prefill_bf16x3(const float* q, const float* kCache, const float* vCache, float* out, int C,
                                   int P, cudaStream_t stream) {
  Problem p{};
  const int rc = prepare(q, kCache, vCache, out, C, P, &p);
  if (rc != ATTN_OK || C == 0) return rc;
  return launch_tc_bf16x3(p, stream);
}

extern "C" int attn_prefill_bf16kv(const float* q, const uint16_t* kCache, const uint16_t* vCache, float* out,
                                   int C, int P, cudaStream_t stream) {
  Problem p{};
  const int rc = prepare(q, reinterpret_cast<const float*>(kCache), reinterpret_cast<const float*>(vCache), out,
                         C, P, &p);
  if (rc != ATTN_OK || C == 0) return rc;
  return launch_tc_bf16(p, stream);
}

extern "C" int attn_full_causal(const float* q, const float* k, const float* v, float* out, int T,
                                cudaStream_t stream) {
  return attn_prefill(q, k, v, out, T, 0, stream);
}

extern "C" int attn_prefill_ffma(const float* q, const float* kCache, const float* vCache,
                                 float* out, int C, int P, cudaStream_t stream) {
  Problem p{};
  const int rc = prepare(q, kCache, vCache, out, C, P, &p);
  if (rc != ATTN_OK || C == 0) return rc;
  return from_cuda(launch_ffma(p, stream));
}

extern "C" int attn_reference_prefill(const float* q, const float* kCache, const float* vCache,
                                      float* out, int C, int P, cudaStream_t stream) {
  Problem p{};
  const int rc = prepare(q, kCache, vCache, out, C, P, &p);
  if (rc != ATTN_OK || C == 0) return rc;
  return from_cuda(launch_reference(p, stream));
}

extern "C" int attn_prefill_paged(const float* q, const float* kPages, const float* vPages,
                                  const int* blockTable, float* out, int C, int P, int numPages,
                                  cudaStream_t stream) {
  Problem p{};
  const int rc = prepare(q, kPages, vPages, out, C, P, &p);
  if (rc != ATTN_OK || C == 0) return rc;
  if (!blockTable || numPages < 1) return ATTN_EINVAL;
  if ((reinterpret_cast<uintptr_t>(blockTable) & 3u) != 0) return ATTN_EALIGN;
  if (numPages > ATTN_MAX_TOKENS / ATTN_PAGE) return ATTN_ERANGE;
  return launch_tc_paged(p, blockTable, numPages, stream);
}

extern "C" size_t attn_decode_workspace_bytes(int B, int maxContext, int numSplits) {
  if (B <= 0 || maxContext < 0 || numSplits < 0) return 0;
  int slots = 0;
  if (decode_slots(&slots) != ATTN_OK) return 0;
  int split_len = 0;
  const int splits = decode_splits(B, maxContext, numSplits, slots, &split_len);
  return decode_workspace_bytes(B, splits);
}

namespace attn {
namespace {
int decode_paged(const float* q, const float* kPages, const float* vPages, const int* blockTable,
                 const int* contextLens, float* out, int B, int maxBlocks, int numPages, int maxContext,
                 int numSplits, void* workspace, size_t workspaceBytes, cudaStream_t stream, int fault) {
  int rc = decode_shape_ok(B, maxBlocks, numPages, maxContext, numSplits);
  if (rc != ATTN_OK || B == 0) return rc;
  if (!q || !kPages || !vPages || !blockTable || !contextLens || !out) return ATTN_EINVAL;
  if (!aligned16(q) || !aligned16(kPages) || !aligned16(vPages) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(blockTable) & 3u) || (reinterpret_cast<uintptr_t>(contextLens) & 3u))
    return ATTN_EALIGN;
  DeviceState* st = nullptr;
  rc = current_device(&st);
  if (rc != ATTN_OK) return rc;
  int slots = 0;
  if ((rc = decode_slots(&slots)) != ATTN_OK) return rc;
  int split_len = 0;
  const int splits = decode_splits(B, maxContext, numSplits, slots, &split_len);
  const size_t need = decode_workspace_bytes(B, splits);
  if (need > 0) {
    if (!workspace || workspaceBytes < need) return ATTN_ESPACE;
    if (!aligned16(workspace)) return ATTN_EALIGN;
  }
  return launch_decode(q, kPages, vPages, blockTable, contextLens, out, static_cast<float*>(workspace), B, maxBlocks,
                       numPages, maxContext, split_len, splits, st->err, stream, fault);
}
}  // namespace
}  // namespace attn

extern "C" int attn_decode_paged(const float* q, const float* kPages, const float* vPages,
                                 const int* blockTable, const int* contextLens, float* out, int B,
                                 int maxBlocks, int numPages, int maxContext, int numSplits, void* workspace,
                                 size_t workspaceBytes, cudaStream_t stream) {
  return decode_paged(q, kPages, vPages, blockTable, contextLens, out, B, maxBlocks, numPages, maxContext, numSplits,
                      workspace, workspaceBytes, stream, 0);
}

extern "C" int attn_selftest_decode_timeout(const float* q, const float* kPages, const float* vPages,
                                            const int* blockTable, const int* contextLens, float* out, int B,
                                            int maxBlocks, int numPages, int maxContext, int numSplits,
                                            void* workspace, size_t workspaceBytes, cudaStream_t stream) {
  if (B < 1 || maxContext < 1) return ATTN_EINVAL;  // no tile, nothing to withhold
  return decode_paged(q, kPages, vPages, blockTable, contextLens, out, B, maxBlocks, numPages, maxContext, numSplits,
                      workspace, workspaceBytes, stream, 1);
}

extern "C" int attn_decode_paged_noalloc(const float* q, const float* kPages, const float* vPages,
                                         const int* blockTable, const int* contextLens, float* out, int B,
                                         int maxBlocks, int numPages, int maxContext, int numSplits,
                                         cudaStream_t stream) {
  static_assert(kDecodeScratchBytes == ATTN_DECODE_SCRATCH_BYTES, "scratch size and header disagree");
  int rc = decode_shape_ok(B, maxBlocks, numPages, maxContext, numSplits);
  if (rc != ATTN_OK || B == 0) return rc;
  if (!q || !kPages || !vPages || !blockTable || !contextLens || !out) return ATTN_EINVAL;
  if (!aligned16(q) || !aligned16(kPages) || !aligned16(vPages) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(blockTable) & 3u) || (reinterpret_cast<uintptr_t>(contextLens) & 3u))
    return ATTN_EALIGN;
  DeviceState* st = nullptr;
  rc = current_device(&st);
  if (rc != ATTN_OK) return rc;
  int slots = 0;
  if ((rc = decode_slots(&slots)) != ATTN_OK) return rc;
  int split_len = 0;
  const int splits = decode_splits(B, maxContext, numSplits, slots, &split_len);
  if (decode_workspace_bytes(B, splits) > kDecodeScratchBytes) return ATTN_ESCRATCH;
  float* scratch = nullptr;
  if (decode_scratch(&scratch) != cudaSuccess) return ATTN_ECUDA;
  return launch_decode(q, kPages, vPages, blockTable, contextLens, out, scratch, B, maxBlocks, numPages, maxContext,
                       split_len, splits, st->err, stream);
}

extern "C" size_t attn_naive_workspace_bytes(int C, int P) {
  if (C < 0 || P < 0 || (long long)P + C > ATTN_MAX_TOKENS) return 0;
  return naive_workspace_bytes(C, P);
}

extern "C" int attn_naive_scores(const float* q, const float* kCache, float* scores, int C, int P,
                                 cudaStream_t stream) {
  DeviceState* st = nullptr;
  const int rc = naive_prepare(C, P, &st);
  if (rc != ATTN_OK || C == 0) return rc;
  if (!q || !kCache || !scores) return ATTN_EINVAL;
  if (!aligned16(q) || !aligned16(kCache) || !aligned16(scores)) return ATTN_EALIGN;
  return from_cuda(launch_naive_scores(q, kCache, scores, C, P, stream));
}

extern "C" int attn_naive_softmax(float* scores, int C, int P, cudaStream_t stream) {
  DeviceState* st = nullptr;
  const int rc = naive_prepare(C, P, &st);
  if (rc != ATTN_OK || C == 0) return rc;
  if (!scores) return ATTN_EINVAL;
  if (!aligned16(scores)) return ATTN_EALIGN;
  return from_cuda(launch_naive_softmax(scores, C, P, stream));
}

extern "C" int attn_naive_weighted_sum(const float* scores, const float* vCache, float* out, int C, int P,
                                       cudaStream_t stream) {
  DeviceState* st = nullptr;
  const int rc = naive_prepare(C, P, &st);
  if (rc != ATTN_OK || C == 0) return rc;
  if (!scores || !vCache || !out) return ATTN_EINVAL;
  if (!aligned16(scores) || !aligned16(vCache) || !aligned16(out)) return ATTN_EALIGN;
  return from_cuda(launch_naive_weighted_sum(scores, vCache, out, C, P, stream));
}

extern "C" int attn_naive_prefill(const float* q, const float* kCache, const float* vCache, float* out,
                                  float* scores, size_t scoresBytes, int C, int P, cudaStream_t stream) {
  DeviceState* st = nullptr;
  int rc = naive_prepare(C, P, &st);
  if (rc != ATTN_OK || C == 0) return rc;
  if (!q || !kCache || !vCache || !out) return ATTN_EINVAL;
  if (!scores || scoresBytes < naive_workspace_bytes(C, P)) return ATTN_ESPACE;
  if (!aligned16(q) || !aligned16(kCache) || !aligned16(vCache) || !aligned16(out) || !aligned16(scores))
    return ATTN_EALIGN;
  if ((rc = from_cuda(launch_naive_scores(q, kCache, scores, C, P, stream))) != ATTN_OK) return rc;
  if ((rc = from_cuda(launch_naive_softmax(scores, C, P, stream))) != ATTN_OK) return rc;
  return from_cuda(launch_naive_weighted_sum(scores, vCache, out, C, P, stream));
}

extern "C" int attn_selftest_timeout(const float* q, const float* kCache, const float* vCache,
                                     float* out, int C, int P, cudaStream_t stream) {
  Problem p{};
  const int rc = prepare(q, kCache, vCache, out, C, P, &p);
  if (rc != ATTN_OK) return rc;
  if (C == 0) return ATTN_EINVAL;
  return launch_tc_fault_test(p, stream);
}

extern "C" int attn_tensor_peak(int bf16, int n, int iters, int ctas, cudaStream_t stream) {
  if ((bf16 != 0 && bf16 != 1) || n < 16 || n > 256 || (n & 15) != 0 || iters < 1 || iters > (1 << 22) ||
      ctas < 1 || ctas > 65535)
    return ATTN_EINVAL;
  DeviceState* st = nullptr;
  const int rc = current_device(&st);
  if (rc != ATTN_OK) return rc;
  return launch_tensor_peak(bf16, n, iters, ctas, st->err, stream);
}

extern "C" int attn_get_device_error(void) {
  DeviceState* st = nullptr;
  const int rc = current_device(&st);
  if (rc != ATTN_OK) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return ATTN_ECUDA;
  unsigned word = 0;
  const unsigned zero = 0;
  if (cudaMemcpyFromSymbol(&word, g_error_word, sizeof(word)) != cudaSuccess) return ATTN_ECUDA;
  if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) return ATTN_ECUDA;
  if (word == kDevErrTimeout) return ATTN_ETIMEOUT;
  if (word == kDevErrBounds) return ATTN_EBOUNDS;
  return word == 0 ? ATTN_OK : ATTN_ECUDA;
}

extern "C" const char* attn_strerror(int code) {
  switch (code) {
    case ATTN_OK: return "success";
    case ATTN_EINVAL: return "invalid argument (a NULL pointer, or a size below what the call accepts)";
    case ATTN_EALIGN: return "a tensor pointer is not 16-byte aligned";
    case ATTN_ERANGE:
      return "a size is out of range (C or P + C above ATTN_MAX_TOKENS, numPages above ATTN_MAX_TOKENS / 16, "
             "B above 65535, or maxContext above 16 * maxBlocks)";
    case ATTN_ELAUNCH: return "kernel launch failed";
    case ATTN_ETIMEOUT: return "a device-side bounded wait expired";
    case ATTN_EBOUNDS: return "a device-side bounds check failed";
    case ATTN_EDEVICE: return "the current device is not sm_103 (GB300)";
    case ATTN_ETMA: return "a TMA tensor map could not be encoded";
    case ATTN_ECUDA: return "a CUDA runtime call failed";
    case ATTN_ESPACE: return "the workspace is missing or smaller than attn_decode_workspace_bytes()";
    case ATTN_ESCRATCH:
      return "the decode partials exceed the library's fixed scratch (ATTN_DECODE_SCRATCH_BYTES): "
             "use fewer splits or attn_decode_paged with a workspace";
    default: return "unknown error code";
  }
}

extern "C" const char* attn_version(void) {
  return "libattnprefill: tcgen05 split-TF32 prefill (contiguous and paged), tcgen05 bf16-K/V prefill, split-KV GQA decode, FFMA, score-matrix and reference kernels, sm_103a";
}
