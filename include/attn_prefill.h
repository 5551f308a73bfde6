/*
 * attn_prefill.h -- C ABI of libattnprefill.so: causal grouped-query flash
 * attention of a prefill chunk against a cached prefix, for sm_103a (GB300).
 *
 * The operation ("Inference Attention 2: Flash Prefill Against a Cached
 * Prefix", Lesson). A chunk of C new tokens at positions P .. P+C-1 attends to
 * the cached keys and values at positions 0 .. P+C-1, causally: chunk row i
 * sees keys j <= P + i. With 32 query heads, 8 KV heads and head dimension 64,
 * query head h reads KV head h / 4, the scale is exactly 1/8, and
 *
 *   out[i][h][:] = sum_{j <= P+i} softmax_j( q[i][h] . k[j][h/4] / 8 ) * v[j][h/4][:]
 *
 * Layouts (attention-v1 contract, same page): fp32, row-major, contiguous:
 *   q       [C][32][64]       the chunk's queries
 *   kCache  [P + C][8][64]    keys of the whole visible sequence
 *   vCache  [P + C][8][64]    values of the whole visible sequence
 *   out     [C][32][64]       written, never read (it may hold garbage or NaN)
 *
 * Ownership. Every pointer is a DEVICE pointer owned by the caller, on the
 * current CUDA device, except the host buffers of the three *_host entry
 * points (described with them). The library allocates no device memory per
 * call. The
 * prefill entry points take no workspace: there is no score matrix anywhere
 * (the contract has no workspace argument). q, kCache and vCache are only
 * read. Two families outside that contract take a caller-owned workspace,
 * described with them: split-KV decode (its segment partials) and the
 * score-matrix pipeline (the matrix itself).
 *
 * Execution. Every compute entry point validates its arguments on the host,
 * enqueues its kernel(s) on `stream` and returns; completion is observed by
 * synchronising the stream. A NULL stream is the legacy default stream.
 * Calls on different streams may overlap; each call reads only its inputs and
 * writes only its out (and its own workspace), except attn_decode_paged_noalloc,
 * whose calls share one library buffer. The first call on a device performs a
 * one-time set-up (device check, kernel attributes), safe from several host
 * threads at once.
 *
 * Errors. 0 means enqueued. A negative return is one of ATTN_E* below and
 * means nothing was enqueued (argument errors) or the launch failed. A kernel
 * that detects an internal fault (a bounded wait that expired, a bounds check
 * that failed) records it in a device-side error word instead of trapping;
 * attn_get_device_error() reads and clears that word. There is no CPU
 * fallback and no alternative back end: on a device that is not sm_103 the
 * entry points return ATTN_EDEVICE.
 *
 * Sizes. 0 <= C <= ATTN_MAX_TOKENS, 0 <= P, P + C <= ATTN_MAX_TOKENS. C == 0
 * is a valid empty call: nothing is read, written or launched and the
 * pointers may be NULL. Pointers must be 16-byte aligned.
 */
#ifndef ATTN_PREFILL_H
#define ATTN_PREFILL_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN_HQ 32
#define ATTN_HKV 8
#define ATTN_D 64
#define ATTN_MAX_TOKENS (1 << 24)
#define ATTN_PAGE 16        /* tokens per page of a paged K/V cache */

/* Return codes. */
#define ATTN_OK 0
#define ATTN_EINVAL -1      /* NULL pointer with C > 0, C < 0, P < 0 */
#define ATTN_EALIGN -2      /* a pointer is not 16-byte aligned */
#define ATTN_ERANGE -3      /* a size out of range: C or P + C above ATTN_MAX_TOKENS, or as a call states */
#define ATTN_ELAUNCH -4     /* the kernel launch failed (cudaGetLastError) */
#define ATTN_ETIMEOUT -5    /* device word: a bounded wait expired */
#define ATTN_EBOUNDS -6     /* device word: a device-side bounds check failed */
#define ATTN_EDEVICE -7     /* the current device is not sm_103 */
#define ATTN_ETMA -8        /* a TMA tensor map could not be encoded */
#define ATTN_ECUDA -9       /* another CUDA runtime call failed */
#define ATTN_ESPACE -10     /* a workspace is missing or too small */
#define ATTN_ESCRATCH -11   /* the decode partials exceed ATTN_DECODE_SCRATCH_BYTES */

/* Size of the fixed device scratch behind attn_decode_paged_noalloc. */
#define ATTN_DECODE_SCRATCH_BYTES (4u << 20)

/*
 * attn_prefill -- the main path: a persistent, warp-specialised tcgen05
 * kernel. A CTA owns a work unit of 32 chunk positions x the 4 query heads of
 * one KV head (GQA packing, "FlashAttention and inference kernels", GQA read
 * amplification exercise), so each K/V tile is staged in shared memory once
 * per group (page 1, Lesson: stage each K/V tile once, reuse it across a
 * resident tile of query rows). Tiles past the causal edge are never loaded
 * and the diagonal tile is masked ("FlashAttention and inference kernels",
 * How FlashAttention evolved: the causal mask). The online softmax carries
 * m, l and the accumulator across tiles and divides once at the end (page 1,
 * Lesson, the tile update). QK^T and PV run on the tensor cores as
 * error-compensated split-TF32: each fp32 operand x = hi + lo with hi exactly
 * representable in tf32, and each product accumulates hi*hi + hi*lo + lo*hi in
 * fp32, so the result matches exact fp32 products to about 2^-20 relative.
 * When the last round of units would leave at least half of the SMs idle and
 * every unit sees 1024 keys or more, a second grid of CTA clusters takes those
 * units, each cluster splitting one along its keys and merging the partials
 * with the split-K rule (same page, Flash-Decoding and the split-K merge):
 * clusters of two, or of three, four or eight when the device holds one such
 * cluster for every unit of that round (a last round of up to twice as many
 * units as clusters of three it holds, each seeing 8192 keys or more, goes
 * to clusters of three in two waves); a chunk with at most half as
 * many units as SMs and a longest unit of 256 keys or more runs as that split
 * grid alone, over clusters of four CTAs (each a quarter of a unit's keys)
 * when the device holds a cluster of four for every unit (chunks of up to 128
 * rows on 152 SMs), or of eight (twelve from 8192 keys) when it holds such a
 * cluster for every unit and the longest sees 1024 keys or more (chunks of up
 * to 32 rows; up to 64 rows over twelves in two waves from 16384 keys), or
 * of three when it holds a cluster of three for every unit (chunks of up to
 * 184 rows); a chunk of up to twice as many units as that, whose longest unit
 * sees 4096 keys or more (8192 for the bf16 paths), splits every unit over
 * three CTAs too, the clusters running in two waves. None of it needs device
 * memory.
 */
int attn_prefill(const float *q, const float *kCache, const float *vCache, float *out,
                 int C, int P, cudaStream_t stream);

/*
 * attn_prefill_bf16x3 -- attn_prefill (fp32 cache, same arguments, layouts and
 * errors) on the bf16 tensor-core path: each fp32 operand is carried as two
 * bf16 terms x = x1 + x2 (x1 rounded to nearest, x2 the rounded remainder) and
 * each product keeps x1 y1 + x1 y2 + x2 y1 in fp32, dropping x2 y2 (below
 * 2^-15 of |x y|). The K/V split runs in shared memory, in place, on each tile
 * as it lands; V needs no transpose.
 */
int attn_prefill_bf16x3(const float *q, const float *kCache, const float *vCache, float *out,
                        int C, int P, cudaStream_t stream);

/*
 * attn_prefill_bf16kv -- attn_prefill with the K/V cache held in bf16, the
 * production cache precision ("FlashAttention and inference kernels",
 * inference: the KV cache in BF16). kCache and vCache are [P + C][8][64] bf16
 * values given as their 16-bit patterns (uint16_t; sign, 8 exponent bits, 7
 * fraction bits); q and out are fp32 as for attn_prefill. The result is the
 * attention over the stored bf16 keys and values to the fp32 tolerance of
 * attn_prefill: K and V enter the tcgen05 kind::f16 MMAs exactly as stored,
 * while q and the probabilities are each split into two bf16 terms (16
 * significant bits together) whose products are accumulated in fp32. Half the
 * K/V bytes of attn_prefill and no conversion pass. Same sizes, alignment and
 * errors as attn_prefill.
 */
int attn_prefill_bf16kv(const float *q, const uint16_t *kCache, const uint16_t *vCache, float *out,
                        int C, int P, cudaStream_t stream);

/*
 * attn_prefill_host, attn_prefill_bf16x3_host, attn_prefill_bf16kv_host --
 * attn_prefill, attn_prefill_bf16x3 and attn_prefill_bf16kv starting and
 * ending in host memory. The call copies q, kCache and vCache from the host
 * buffers into the caller's device buffers, computes, and copies out back to
 * the host. It applies the chunked-prefill identity one level up ("Inference
 * Attention 2: Flash Prefill Against a Cached Prefix", Lesson: a chunk at
 * positions P .. P+C-1 attends to every position up to its own): rows r0 ..
 * r1-1 of the result are the prefill of those query rows against positions
 * 0 .. P+r1-1. So the chunk runs as sub-chunks of whole 32-row query tiles,
 * each one full round of units (SMs / 8 tiles: 608 rows on 152 SMs, the last
 * the remainder; at most four, equal ones beyond that), and each copies in
 * only its own query rows and the K/V rows the sub-chunk before it did not
 * need. Copy-in of sub-chunk s+1 and copy-out of sub-chunk s-1 run under the
 * compute of sub-chunk s, on two copy streams the library keeps per device,
 * and consecutive sub-chunks compute alternately on `stream` and on a third
 * library stream, so a sub-chunk's blocks take SMs as the previous one's
 * finish (serving chunk end to end: 0.351 -> 0.325 ms). Each sub-chunk's rows are exactly
 * those of the device-pointer entry point called on that sub-chunk; against one
 * call on the whole chunk they agree to rounding (that call may split its last
 * round's units over CTA clusters, another summation order).
 *
 *   q_host, kCache_host, vCache_host   read; the layouts of attn_prefill
 *                                      (uint16_t bf16 patterns for the
 *                                      bf16kv cache)
 *   out_host                           written
 *   q_dev, kCache_dev, vCache_dev,     the caller's device buffers with the
 *   out_dev                            same layouts; all four are written
 *                                      (after a completed call they hold the
 *                                      inputs and the result)
 *
 * Host memory should be page-locked (cudaHostAlloc or cudaHostRegister):
 * pageable buffers are accepted but each of their copies then blocks the
 * calling thread, so nothing overlaps. The copies use cudaMemcpyDefault, so
 * any memory the driver can copy from or to is accepted.
 * Ordering. The copies start after the work enqueued on `stream` before the
 * call, and `stream` waits for the last copy-out: synchronising `stream`
 * observes out_host complete. Calls from several host threads are serialised
 * while they enqueue (the library's per-device streams and events are shared).
 * Set-up. The first call on a device creates three non-blocking streams and
 * ten events (no device memory); they live until the process ends.
 * Errors: those of the device-pointer entry point for the device buffers and
 * sizes; ATTN_EINVAL for a NULL host pointer with C > 0; ATTN_ECUDA when a copy
 * or a stream or event call fails. After an error, copies may already have
 * been enqueued; `stream` still waits for every one of them.
 */
int attn_prefill_host(const float *q_host, const float *kCache_host, const float *vCache_host,
                      float *out_host, float *q_dev, float *kCache_dev, float *vCache_dev, float *out_dev,
                      int C, int P, cudaStream_t stream);
int attn_prefill_bf16x3_host(const float *q_host, const float *kCache_host, const float *vCache_host,
                             float *out_host, float *q_dev, float *kCache_dev, float *vCache_dev, float *out_dev,
                             int C, int P, cudaStream_t stream);
int attn_prefill_bf16kv_host(const float *q_host, const uint16_t *kCache_host, const uint16_t *vCache_host,
                             float *out_host, float *q_dev, uint16_t *kCache_dev, uint16_t *vCache_dev,
                             float *out_dev, int C, int P, cudaStream_t stream);

/*
 * attn_prefill_paged -- attn_prefill against a paged K/V cache ("FlashAttention
 * and inference kernels", PagedAttention: a cache is cut into fixed pages and a
 * block table maps the i-th logical page to its physical page, so the kernel
 * gains one indirection per K/V read). Token t's key and value live in slot
 * t % 16 of physical page blockTable[t / 16]:
 *   kPages, vPages  [numPages][16][8][64] fp32, device pointers
 *   blockTable      int32 device array of at least ceil((P + C) / 16) entries,
 *                   each in [0, numPages); pages may be shared and in any order
 * q and out as for attn_prefill. Slots of a page past position P + C - 1 are
 * never given weight and may hold any values, NaN included. An entry outside
 * [0, numPages) is read as zeros and recorded as ATTN_EBOUNDS in the device
 * error word (see attn_get_device_error). Errors: ATTN_EINVAL for a NULL table
 * or numPages < 1, ATTN_EALIGN for a table not 4-byte aligned, ATTN_ERANGE for
 * numPages > ATTN_MAX_TOKENS / 16, otherwise as attn_prefill.
 */
int attn_prefill_paged(const float *q, const float *kPages, const float *vPages,
                       const int *blockTable, float *out, int C, int P, int numPages,
                       cudaStream_t stream);

/*
 * attn_decode_paged -- one decode step for B sequences: the chunk of one token
 * (page 1, Lesson: the same formula at one row is decode, bandwidth-bound).
 * Sequence b has one query per head, q[b][h][:], whose own key and value are
 * already in the cache at position contextLens[b] - 1; it attends to keys
 * 0 .. contextLens[b] - 1 with scale 1/8, query head h reading KV head h / 4:
 *   out[b][h][:] = sum_{j < ctx_b} softmax_j(q[b][h] . k_b[j][h/4] / 8) v_b[j][h/4][:]
 * The cache is paged ("FlashAttention and inference kernels", PagedAttention):
 *   kPages, vPages  [numPages][16][8][64] fp32
 *   blockTable      int32 [B][maxBlocks]: sequence b's token t is slot t % 16
 *                   of page blockTable[b * maxBlocks + t / 16]
 *   contextLens     int32 [B], each in [0, maxContext] (0 gives zeros)
 *   q, out          [B][32][64] fp32
 * A block owns (key segment, KV head, sequence) and all four query heads of
 * that KV head, so each K/V row is read once per group; segments are merged
 * with m = max m_s, w_s = e^(m_s - m) l_s, out = sum w_s O_s / sum w_s (same
 * page, Flash-Decoding / split-K merge), skipping empty segments.
 * numSplits: segments per sequence, 0 = chosen from B, maxContext and how many
 * split blocks the device holds at once (segments of at least 256 keys, as
 * many as fill those slots best). With more than one segment the partials need `workspace`, a device
 * buffer of at least attn_decode_workspace_bytes(B, maxContext, numSplits)
 * bytes, 16-byte aligned, owned by the caller, overwritten by the call, not
 * used after the call's kernels finish. Errors: ATTN_EINVAL (NULL pointer,
 * negative size, maxBlocks or numPages < 1), ATTN_ERANGE (B > 65535,
 * maxContext > 16 * maxBlocks, sizes above ATTN_MAX_TOKENS), ATTN_EALIGN,
 * ATTN_ESPACE (workspace missing or too small), ATTN_ETMA (the page pools'
 * tensor maps could not be encoded). A context length outside
 * [0, maxContext] or a page index outside [0, numPages) is recorded as
 * ATTN_EBOUNDS in the device error word and clamped / read as zeros. B == 0 is
 * a no-op.
 */
int attn_decode_paged(const float *q, const float *kPages, const float *vPages, const int *blockTable,
                      const int *contextLens, float *out, int B, int maxBlocks, int numPages,
                      int maxContext, int numSplits, void *workspace, size_t workspaceBytes,
                      cudaStream_t stream);

/*
 * attn_decode_workspace_bytes -- the workspace attn_decode_paged needs for the
 * same (B, maxContext, numSplits) on the current device; 0 when one segment
 * per sequence suffices (or for invalid arguments).
 */
size_t attn_decode_workspace_bytes(int B, int maxContext, int numSplits);

/*
 * attn_decode_paged_noalloc -- attn_decode_paged without a workspace argument,
 * for callers that cannot hand the library any device memory: a serving loop
 * whose buffers are all planned once at start-up, a C host that has no access
 * to the device allocator of the framework that owns the GPU, or a
 * latency-critical path where a cudaMalloc (which may synchronise the device)
 * is not allowed. The pages describe no such variant; it exists for those
 * callers only and computes exactly what attn_decode_paged computes with the
 * same numSplits.
 *
 * The segment partials go to one fixed buffer of ATTN_DECODE_SCRATCH_BYTES
 * (4 MiB) that is part of the library's device image, so the call allocates
 * nothing, neither here nor in any library it calls. That buffer holds
 * B * 8 * splits records of 1056 bytes. The automatic split count (numSplits =
 * 0) weighs fill against waves of the device's resident split blocks (its
 * slot count: SMs x the blocks per SM the occupancy query reports, 3 x 152 =
 * 456 on a GB300); when it splits at all, B * 8 * splits stays at or below 7
 * slot counts (a sweep of B = 1 .. 65535 and maxContext = 256 .. 2^24), i.e.
 * at most 3192 records, 3.2 MiB, on a GB300, so automatic calls fit there. A
 * call whose partials would not fit (a large explicit numSplits with many
 * sequences) returns ATTN_ESCRATCH and enqueues nothing; one segment per
 * sequence uses no scratch at all.
 *
 * Sharing. All calls on a device use the same buffer, which keeps whatever the
 * last call left there (nothing in it needs to start at zero: each call writes
 * every record it reads). Two calls that can run at the same time, on
 * different streams or from different host threads without ordering between
 * them, race on it and may return wrong results: order them on one stream or
 * use attn_decode_paged with a workspace each.
 *
 * Set-up. The first call on a device, with that device current, looks up the
 * buffer's device address (cudaGetSymbolAddress) and caches it; make that
 * first call before any stream capture. Arguments, layouts and other errors as
 * attn_decode_paged; ATTN_ECUDA if the address lookup fails.
 */
int attn_decode_paged_noalloc(const float *q, const float *kPages, const float *vPages,
                              const int *blockTable, const int *contextLens, float *out, int B,
                              int maxBlocks, int numPages, int maxContext, int numSplits,
                              cudaStream_t stream);

/*
 * The score-matrix pipeline ("Inference Attention 1: The Full Score Matrix",
 * Lesson): attention as an eager framework runs it, three kernels with the
 * whole score matrix in global memory between them. It is the in-run measure
 * of what that matrix costs; attn_prefill computes the same result without it.
 *
 *   scores  [32][C][P + C] fp32, device, owned by the caller: row i of head h
 *           at scores + (h * C + i) * (P + C), 16-byte aligned,
 *           attn_naive_workspace_bytes(C, P) bytes (32 x T x T floats for a
 *           full prompt of T tokens: 512 MiB at T = 2048).
 *
 * attn_naive_scores writes q[i][h] . k[j][h/4] / 8 for j <= P + i and -inf
 * above the diagonal; attn_naive_softmax replaces each row in place by its
 * softmax (maximum subtracted first; 0 above the diagonal); attn_naive_weighted_sum
 * writes out[i][h][:] = sum_j scores[h][i][j] v[j][h/4][:]. attn_naive_prefill
 * runs the three in order on `stream` and returns ATTN_ESPACE if scoresBytes is
 * too small. q, kCache, vCache and out are as for attn_prefill. Errors as
 * attn_prefill, plus ATTN_ERANGE for C above 4,194,240 (the grid's row limit).
 * C == 0 is a no-op. attn_naive_workspace_bytes returns 0 for invalid sizes.
 */
size_t attn_naive_workspace_bytes(int C, int P);
int attn_naive_scores(const float *q, const float *kCache, float *scores, int C, int P,
                      cudaStream_t stream);
int attn_naive_softmax(float *scores, int C, int P, cudaStream_t stream);
int attn_naive_weighted_sum(const float *scores, const float *vCache, float *out, int C, int P,
                            cudaStream_t stream);
int attn_naive_prefill(const float *q, const float *kCache, const float *vCache, float *out,
                       float *scores, size_t scoresBytes, int C, int P, cudaStream_t stream);

/*
 * attn_full_causal -- a whole prompt with nothing cached: identical to
 * attn_prefill(q, k, v, out, T, 0, stream) ("Inference Attention 1: The Full
 * Score Matrix", Lesson: q [T][32][64], k and v [T][8][64], row i sees j <= i).
 */
int attn_full_causal(const float *q, const float *k, const float *v, float *out,
                     int T, cudaStream_t stream);

/*
 * attn_prefill_ffma -- the same operation on the FP32 CUDA cores (FFMA), with
 * the same GQA-packed tiling but plain shared-memory staging. Exact fp32
 * products; kept as the precision reference for the tensor-core path and as
 * the fallback design. Same arguments, layouts and errors as attn_prefill.
 */
int attn_prefill_ffma(const float *q, const float *kCache, const float *vCache, float *out,
                      int C, int P, cudaStream_t stream);

/*
 * attn_reference_prefill -- the page's starter design rebuilt as the in-run
 * timing reference (page 1, Starter code): one warp per (chunk row, query
 * head), every row walking its whole K/V prefix through the memory system,
 * rescaling by exp(m_old - m_new) at every key. Correct and slow by design.
 * Same arguments, layouts and errors as attn_prefill.
 */
int attn_reference_prefill(const float *q, const float *kCache, const float *vCache, float *out,
                           int C, int P, cudaStream_t stream);

/*
 * attn_selftest_timeout -- a test of the failure path, not a computation. It
 * launches the attn_prefill kernel with one K tile deliberately never loaded
 * and every bounded wait limited to 20 ms, so a wait expires: the kernel
 * records ATTN_ETIMEOUT in the device error word, winds down all its warps,
 * frees its tensor memory and returns; the context stays usable. `out` is left
 * unspecified. Requires C >= 1 (ATTN_EINVAL otherwise). Returns 0 once enqueued;
 * the caller then reads the outcome with attn_get_device_error().
 */
int attn_selftest_timeout(const float *q, const float *kCache, const float *vCache, float *out,
                          int C, int P, cudaStream_t stream);

/*
 * attn_selftest_decode_timeout -- the same test for the decode kernel: the
 * arguments, checks and workspace of attn_decode_paged, but every split block
 * posts the bytes of its first K/V tile without ever loading it and every
 * bounded wait is limited to 20 ms, so each block's wait expires; the block
 * records ATTN_ETIMEOUT, gives the copies it did issue a bounded wait and
 * returns without writing. `out` is left unspecified and the context stays
 * usable. Requires B >= 1 and maxContext >= 1 (ATTN_EINVAL otherwise); a
 * sequence with context 0 has no tile and returns normally.
 */
int attn_selftest_decode_timeout(const float *q, const float *kPages, const float *vPages, const int *blockTable,
                                 const int *contextLens, float *out, int B, int maxBlocks, int numPages,
                                 int maxContext, int numSplits, void *workspace, size_t workspaceBytes,
                                 cudaStream_t stream);

/*
 * attn_tensor_peak -- a measurement of this GPU's tensor pipe, not an
 * attention computation: the rate against which the prefill kernels'
 * contractions are judged compute-bound or not (page 1, "Inference Attention
 * 2: Flash Prefill Against a Cached Prefix", What you will learn: read SM
 * throughput to decide what bounds a kernel). Launches `ctas` CTAs (one per
 * SM when ctas <= SMs); each issues `iters` dense tcgen05.mma instructions of
 * M = 128, N = n back to back from shared-memory operands holding
 * pseudo-random values, K = 8 tf32 elements (bf16 = 0: kind::tf32) or K = 16
 * bf16 elements (bf16 = 1: kind::f16), fp32 accumulation in tensor memory.
 * One launch performs ctas * iters * 2 * 128 * n * K flops; time it with
 * events on `stream`. Nothing is read or written outside the CTAs' own
 * shared and tensor memory; no device memory is allocated. Arguments: bf16
 * 0 or 1, n a multiple of 16 in [16, 256], iters in [1, 2^22], ctas in
 * [1, 65535] (ATTN_EINVAL otherwise). An expired completion wait (2 s) is
 * recorded as ATTN_ETIMEOUT in the device error word.
 */
int attn_tensor_peak(int bf16, int n, int iters, int ctas, cudaStream_t stream);

/*
 * attn_get_device_error -- synchronises the current device, then returns and
 * clears the device-side error word: 0, ATTN_ETIMEOUT or ATTN_EBOUNDS (the
 * first fault recorded since the last call), or ATTN_ECUDA if the
 * synchronisation itself failed.
 */
int attn_get_device_error(void);

/* attn_strerror -- a static, human-readable string for any return code. */
const char *attn_strerror(int code);

/* attn_version -- a static string naming the build (kernels and arch). */
const char *attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_PREFILL_H */
