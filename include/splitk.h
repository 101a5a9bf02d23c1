/*
 * splitk.h -- C ABI of the GB300 (sm_103a) split-K BF16 decode GEMM.
 *
 *     C[l][m][n] = bf16_rne( sum_k A[l][n][k] * B[l][m][k] )
 *
 * Operation (the vLLM API page of module
 * vllm.models.kimi_k3.nvidia.specialized_decode.cutedsl.gemm.splitk,
 * class SplitKGemm and its module docstring): a BF16 GEMM whose K dimension is
 * split across the CTAs of one thread-block cluster.  Each cluster rank
 * accumulates an exact, contiguous K slice in FP32 (tensor memory); the peer
 * ranks publish their FP32 partials to rank 0's shared memory; rank 0 adds
 * them in rank order, converts once to BF16 (round to nearest even) and
 * stores.  Operands are "swapped": the weight rows (public N) run along the
 * 128-wide MMA M dimension and the few tokens (public M) along MMA N.
 *
 * Layouts (all row-major, compact, L outermost, bf16 = 2 bytes):
 *   A  [L][N][K]  weights ("kernel A, K-major"), K contiguous
 *   B  [L][M][K]  token activations, K contiguous
 *   C  [L][M][N]  output, N contiguous
 *
 * Ownership: the caller owns A, B, C and the stream.  The library owns only
 * its caches: device-resident CUDA tensor maps of A (128 bytes each, one per
 * distinct (A pointer, N, K, L)) in a device pool allocated on first use, a
 * pinned host mirror of that pool, and host-side tensor maps of B.
 * splitk_release() frees them.
 *
 * Execution: every call is asynchronous on `stream` and returns after the
 * enqueue.  Calls launch with programmatic dependent launch (PDL): the kernel
 * may begin streaming A while the previous kernel on the stream is still
 * running, and waits for that kernel's completion (griddepcontrol.wait)
 * before it reads B or writes C.  So A must not be written by the kernel that
 * immediately precedes the call on the same stream; pass SPLITK_FLAG_NO_PDL
 * to splitk_gemm_bf16_planned() when it is.
 *
 * Errors: every int-returning call returns SPLITK_OK (0) or a negative
 * splitk_status code; no exception crosses the ABI, nothing is printed.
 * Failed argument checks enqueue no work.
 */
#ifndef SPLITK_H
#define SPLITK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define SPLITK_API __declspec(dllexport)
#else
#define SPLITK_API __attribute__((visibility("default")))
#endif

/* A cudaStream_t (struct CUstream_st*).  NULL is the legacy default stream. */
typedef struct CUstream_st *splitk_stream_t;

enum splitk_status {
    SPLITK_OK = 0,
    /* M, N, K or L < 1, a size past a hardware limit (N > 65535 * 128,
       L > 65535, K > 2^31 - 128, or more than 2^31 - 1 CTAs along the
       grid's x), K not a multiple of 8 (TMA row stride), or fewer 128-wide
       K tiles than split ranks. */
    SPLITK_ERR_INVALID_SHAPE = -1,
    /* A or B not 16-byte aligned (TMA), or C not 2-byte aligned. */
    SPLITK_ERR_MISALIGNED = -2,
    /* split_k not in {0 (plan chooses), 1, 2, 4, 8}. */
    SPLITK_ERR_UNSUPPORTED_SPLIT = -3,
    /* No tile / stage configuration fits the shared-memory budget. */
    SPLITK_ERR_NO_FIT = -4,
    /* A CUDA runtime or driver call failed (launch, copy, allocation). */
    SPLITK_ERR_CUDA = -5,
    /* A bounded wait inside the kernel ran out (see splitk_get_fault). */
    SPLITK_ERR_TIMEOUT = -6,
    /* A required pointer argument is NULL. */
    SPLITK_ERR_NULL = -7,
    /* The device tensor-map pool is full; call splitk_release(). */
    SPLITK_ERR_CACHE_FULL = -8,
    /* No CUDA device, or the current device is not compute capability 10.3. */
    SPLITK_ERR_UNSUPPORTED_DEVICE = -9,
    /* A plan passed to splitk_gemm_bf16_planned() does not match the shape. */
    SPLITK_ERR_BAD_PLAN = -10,
    /* splitk_gemm_bf16_noalloc(): the call needs more scratch than its
       static array holds. */
    SPLITK_ERR_SCRATCH = -11,
    /* splitk_gemm_bf16_zerocopy(): a host buffer is not page-locked and
       mapped into the device address space. */
    SPLITK_ERR_NOT_MAPPED = -12,
    /* splitk_gemm_bf16_noalloc(): the stream is capturing a CUDA graph. */
    SPLITK_ERR_CAPTURE = -13
};

/* Flags of splitk_gemm_bf16_planned(). */
#define SPLITK_FLAG_NO_PDL 0x1u

/* Weight formats (splitk_plan_t.weight_format). */
#define SPLITK_WEIGHTS_BF16 0        /* A[L][N][K] bf16                              */
#define SPLITK_WEIGHTS_E2M1_E8M0 1   /* A16W4: codes A_q[L][N][K/2], scales A_s[L][N][K/32] */
#define SPLITK_WEIGHTS_E4M3_E8M0 2   /* A16W8: codes A_q[L][N][K], scales A_s[L][N][K/32]   */

/*
 * A launch configuration ("tactic": the page's SplitKTactic fields mma_m,
 * mma_n, ab_stages, split_k, plus what the launcher derives from them).
 */
typedef struct splitk_plan_t {
    int mma_m;             /* 128: weight rows per CTA tile (tcgen05 MMA M)    */
    int mma_n;             /* 16, 32, 64 or 128: token columns per CTA tile    */
    int stages;            /* shared-memory ring depth (2..8)                  */
    int split_k;           /* CTAs per cluster, each owning K/split_k of K     */
    int k_tiles_per_cta;   /* 128-wide K tiles each CTA accumulates            */
    int mailbox_dedicated; /* 1: partials land in their own smem region;
                              0: they reuse rank 0's drained weight ring       */
    int mailbox_quads;     /* 4-column groups of partials per reduction round  */
    int reduce_rounds;     /* rounds of the rank-0 reduction                    */
    unsigned grid[3];      /* (split_k * ceil(M/mma_n), ceil(N/128), L)        */
    unsigned cluster[3];   /* (split_k, 1, 1)                                  */
    size_t smem_bytes;     /* dynamic shared memory per CTA                    */
    int ctas_per_sm;       /* CTAs the smem budget was sized for               */
    int pdl_trigger;       /* when a CTA lets the next kernel on the stream
                              launch: 0 after its last weight TMA issue,
                              1 as soon as it holds its tensor memory          */
    int reduce_scatter;    /* 0: rank 0 sums the whole tile and stores it (the
                              page's design); 1: rank r sums and stores weight
                              rows [r*128/split, (r+1)*128/split) -- same
                              additions in the same order, same bits, 1/split
                              of the DSMEM bytes per SM; needs split_k > 1 and
                              a dedicated mailbox of min(M, mma_n) * 512 B     */
    int b_resident;        /* 0: each activation K tile rides the weight ring
                              stage it is multiplied with (the page's design);
                              1: all of the CTA's activation K tiles have their
                              own buffer and arrive at once after the
                              programmatic-dependent-launch wait               */
    int a_tmem_tiles;      /* 0..3 leading weight K tiles that the MMA warp
                              copies from the ring into tensor memory
                              (tcgen05.cp) before the activations exist, so
                              their stages take further tiles; the MMAs then
                              read those tiles from tensor memory.  Needs
                              b_resident = 1                                   */
    unsigned tmem_cols;    /* tensor-memory columns per CTA (derived: the
                              accumulators, then 64 per staged tile from a
                              64-column boundary, rounded up to a power of
                              two); the CTAs that fit an SM by shared memory
                              never need more than 512                         */
    int mma_issuers;       /* 1: one thread issues every MMA (the page's
                              design); 2: a second thread takes the odd K
                              tiles into its own accumulator, the epilogue
                              adds the two (one more FP32 addition per output,
                              in a fixed order); stages must be a multiple of
                              mma_issuers                                      */
    int b_loader;          /* with b_resident: 0 the activation warp loads the
                              activation tiles by TMA; 1 the 128 epilogue
                              threads load them with 16-byte loads and store
                              them swizzled (for few rows: no TMA queue)       */
    int l2_prefetch;       /* 1: at CTA start, prefetch into L2 the weight K
                              tiles that neither the ring nor tensor memory
                              holds before the programmatic-dependent-launch
                              wait returns                                     */
    int weight_format;     /* SPLITK_WEIGHTS_BF16, or SPLITK_WEIGHTS_E2M1_E8M0
                              (plans of splitk_plan_w4a16*), or
                              SPLITK_WEIGHTS_E4M3_E8M0 (splitk_plan_w8a16*):
                              then `stages` (1..k_tiles_per_cta) is the ring
                              of packed code tiles (all of the CTA's at once
                              when equal), `a_tmem_tiles` (1..3) the TMEM
                              slots the epilogue threads decode tiles into,
                              b_resident = 1, mma_issuers = 1; smem_bytes may
                              exceed the layout's need, which caps how many
                              CTAs share an SM (so the slots fit its TMEM)   */
    int w4_smem_tiles;     /* A16W4 only: 1 = the one K tile after the TMEM
                              slots (k_tiles_per_cta = a_tmem_tiles + 1) is
                              decoded into a 32 KiB bf16 stage in shared
                              memory, so that every tile is decoded before the
                              programmatic-dependent-launch wait returns     */
    int b_stages;          /* persistent plans: 0 = each activation K tile
                              rides the weight ring stage it is multiplied
                              with (`stages` deep); 2..8 = the activations
                              have their own ring of b_stages stages and
                              `stages` is the weight ring's depth alone (at
                              wide tiles an activation stage is as large as a
                              weight stage but comes from L2, so a shallower
                              activation ring leaves shared memory for more
                              weight tiles or for a mailbox that reduces a
                              tile in one round).  0 for every other plan    */
    int persistent;        /* 0: one CTA per (output tile, K rank), the grid
                              above.  1: the persistent kernel: grid
                              (split_k, clusters, 1), each cluster of split_k
                              CTAs (one per SM) walking the output tiles
                              `clusters` apart, its ring running on from tile
                              to tile and its accumulator alternating between
                              two TMEM buffers, so that a tile's reduction
                              overlaps the next tile's loads and MMAs.  Needs
                              split_k >= 2 and the scattered reduction
                              (reduce_scatter = 1, mailbox_dedicated = 1,
                              b_resident = 0, a_tmem_tiles = 0,
                              mma_issuers = 1).  grid[1] is an upper bound: a
                              launch uses at most as many clusters as the
                              device holds at once and as there are tiles   */
    int w4_decoders;       /* A16W4 only (0 for bf16 plans): 1 = the four
                              epilogue warps decode the weight tiles; 2 = four
                              more warps (384 threads a CTA, at most 2 CTAs
                              an SM) decode the second half of every tile's K
                              beside them                                   */
} splitk_plan_t;

/*
 * Picks the tactic for the current CUDA device.  split_k = 0 lets the plan
 * choose among {1, 2, 4, 8}.  Needs a device (SPLITK_ERR_UNSUPPORTED_DEVICE
 * otherwise); writes *out only on success.
 */
SPLITK_API int splitk_plan(int M, int N, int K, int L, int split_k,
                           splitk_plan_t *out);

/*
 * The same choice for a described device, without touching CUDA: num_sms
 * streaming multiprocessors, smem_per_sm bytes of shared memory per SM and
 * smem_per_block_optin bytes at most per CTA.
 */
SPLITK_API int splitk_plan_for(int M, int N, int K, int L, int split_k,
                               int num_sms, size_t smem_per_sm,
                               size_t smem_per_block_optin, splitk_plan_t *out);

/*
 * C = B * A^T with the tactic splitk_plan() picks for (M, N, K, L, split_k).
 * a, b, c are device pointers (layouts above); a and b 16-byte aligned.
 * C is written once (not accumulated); rows m >= M and columns n >= N of the
 * padded tiles are never written.  The first call for a given A pointer and
 * shape encodes A's tensor map and copies it to the device (allocating the
 * pool on the first call of all).  Outside a graph capture that copy is
 * synchronous, so later calls on any stream may use the map; inside a
 * capture it is a node of the graph, and calls on other streams must then
 * wait until the graph has run once.  Make that first call outside any
 * capture.
 */
SPLITK_API int splitk_gemm_bf16(const void *a, const void *b, void *c,
                                int M, int N, int K, int L, int split_k,
                                splitk_stream_t stream);

/*
 * A16W4: C[l][m][n] = bf16_rne( sum_k w(l,n,k) * B[l][m][k] ) with 4-bit
 * weights: w = e2m1(code) * 2^(scale - 127), the Muse Spark AMD dev page's
 * e8m0_f32 and fp4x8_bf16 ("a16w4 decode").
 *   a_q      device, [L][N][K/2] bytes: element k of weight row n in the low
 *            nibble of byte k/2 when k is even ("low nibble first"), 16-byte
 *            aligned.  E2M1 code: sign bit 3, exponent bits 2..1 (bias 1),
 *            mantissa bit 0.
 *   a_scale  device, [L][N][K/32] bytes: one E8M0 code (1..252, 2^(x-127))
 *            per 32 consecutive k of a row, 4-byte aligned.  Codes outside
 *            1..252 are outside the contract and decode as follows: 0 as a
 *            zero scale (the format's value, 2^-127, is not applied), 253
 *            and 254 as 2^126 and 2^127 (weights past bf16's largest finite
 *            value become +-Inf), 255 (not a number in the format) as +Inf
 *            (a zero weight times it is NaN).
 *   b, c     as splitk_gemm_bf16().
 * K must be a multiple of 128, M at most 32, and a CTA's K slice at most 8
 * tiles of 128 (else SPLITK_ERR_INVALID_SHAPE / SPLITK_ERR_NO_FIT).  The
 * weights are decoded to bf16 on chip, exactly, and multiplied by the same
 * tcgen05 BF16 MMA as splitk_gemm_bf16().
 */
SPLITK_API int splitk_plan_w4a16_for(int M, int N, int K, int L, int split_k,
                                     int num_sms, size_t smem_per_sm,
                                     size_t smem_per_block_optin, splitk_plan_t *out);
SPLITK_API int splitk_plan_w4a16(int M, int N, int K, int L, int split_k,
                                 splitk_plan_t *out);
SPLITK_API int splitk_gemm_w4a16(const void *a_q, const void *a_scale, const void *b,
                                 void *c, int M, int N, int K, int L, int split_k,
                                 splitk_stream_t stream);
SPLITK_API int splitk_gemm_w4a16_planned(const void *a_q, const void *a_scale,
                                         const void *b, void *c, int M, int N, int K,
                                         int L, const splitk_plan_t *plan,
                                         unsigned flags, splitk_stream_t stream);

/*
 * A16W8: C[l][m][n] = bf16_rne( sum_k w(l,n,k) * B[l][m][k] ) with 8-bit
 * weights: w = e4m3(code) * 2^(scale - 127).  The element format is E4M3,
 * as the DeepSeek-V4.1 AMD mono ops page's fp8_pack4 packs it ("four E4M3
 * bytes, RNE"): sign bit 7, exponent bits 6..3 (bias 7), mantissa bits 2..0,
 * no infinities, 0x7F / 0xFF not a number, largest finite 448.  The block
 * scale is the one of the 4-bit weights above: one E8M0 code per 32
 * consecutive k of a row.
 *   a_q      device, [L][N][K] bytes, one code per k, 16-byte aligned.
 *   a_scale  device, [L][N][K/32] bytes, 4-byte aligned.  Codes 3..246 keep
 *            every decoded weight a finite bf16 value with no bits below
 *            2^-133 (exact); outside that range the decode saturates or
 *            rounds as bf16 arithmetic does (0 and 255 as for the 4-bit
 *            weights).  The two not-a-number weight codes are outside the
 *            contract: they decode as +-480 times the scale (their bits
 *            placed like those of any other code).
 *   b, c     as splitk_gemm_bf16().
 * K must be a multiple of 128, M at most 32, and a CTA's K slice at most 8
 * tiles of 128 (else SPLITK_ERR_INVALID_SHAPE / SPLITK_ERR_NO_FIT).  The
 * plan carries weight_format = SPLITK_WEIGHTS_E4M3_E8M0; otherwise the plan
 * fields, kernel and tactics are those of the 4-bit weights.
 */
SPLITK_API int splitk_plan_w8a16_for(int M, int N, int K, int L, int split_k,
                                     int num_sms, size_t smem_per_sm,
                                     size_t smem_per_block_optin, splitk_plan_t *out);
SPLITK_API int splitk_plan_w8a16(int M, int N, int K, int L, int split_k,
                                 splitk_plan_t *out);
SPLITK_API int splitk_gemm_w8a16(const void *a_q, const void *a_scale, const void *b,
                                 void *c, int M, int N, int K, int L, int split_k,
                                 splitk_stream_t stream);
SPLITK_API int splitk_gemm_w8a16_planned(const void *a_q, const void *a_scale,
                                         const void *b, void *c, int M, int N, int K,
                                         int L, const splitk_plan_t *plan,
                                         unsigned flags, splitk_stream_t stream);

/*
 * Checks a plan against a shape on a described device without touching CUDA
 * (the check every launch makes): SPLITK_OK, or SPLITK_ERR_BAD_PLAN /
 * INVALID_SHAPE / UNSUPPORTED_SPLIT / NO_FIT.  Useful before handing a
 * hand-made plan to splitk_gemm_bf16_planned().
 */
SPLITK_API int splitk_plan_check_for(const splitk_plan_t *plan, int M, int N,
                                     int K, int L, size_t smem_per_sm,
                                     size_t smem_per_block_optin);

/*
 * Every valid tactic for a shape on a described device, without CUDA:
 * splitk_plan_for()'s choice first (followed, when that is a persistent plan,
 * by the per-tile kernel's own choice), then the page's ring (2-8 stages, one or
 * two MMA issuers, either PDL trigger) and the staged family (resident
 * activations, 0-3 weight tiles in tensor memory, TMA or epilogue-thread
 * activation loads, L2 prefetch), for each split (all valid ones when
 * split_k = 0) and each reduction (rank 0 with its own or an aliased
 * mailbox, scattered), then the persistent kernel at each ring depth that
 * fits (split_k >= 2).  Writes up to max_out plans to out and returns how
 * many exist (call with max_out = 0 to size the array), or a negative
 * status.
 */
SPLITK_API int splitk_plan_candidates_for(int M, int N, int K, int L,
                                          int split_k, int num_sms,
                                          size_t smem_per_sm,
                                          size_t smem_per_block_optin,
                                          splitk_plan_t *out, int max_out);

/*
 * Measures every candidate of splitk_plan_candidates_for() on the current
 * device and returns the fastest in *best (and its time per call in
 * *best_us_per_call, if not null).  Each candidate runs `reps` back-to-back
 * launches on `stream` (programmatic dependent launch on), cycling through
 * the n_a weight tensors a_list[0..n_a-1] of identical shape -- a model's
 * same-shape layers, or copies whose total exceeds the L2 cache, so that the
 * weights stream from HBM as in decoding -- with the same activations b and
 * output c.  Synchronises the stream.  Every launch is checked like
 * splitk_gemm_bf16_planned(); waits that time out are recorded as usual
 * (splitk_get_status()).  A setup-time call: it holds the library's lock
 * for the whole measurement.
 */
SPLITK_API int splitk_tune(const void *const *a_list, int n_a, const void *b,
                           void *c, int M, int N, int K, int L, int split_k,
                           int reps, splitk_stream_t stream, splitk_plan_t *best,
                           float *best_us_per_call);

/*
 * C = B * A^T + bias with the bias added per output feature n in FP32 before
 * the one rounding to bf16: C[l][m][n] = bf16_rne(sum_k A B + bias[l][n]).
 * This is the bias argument of the page's SplitKGemm launcher (left unused
 * there).  bias is a device pointer to [L][N] bf16, 2-byte aligned.  Like A,
 * the bias is read before the programmatic-dependent-launch wait, so it must
 * not be written by the kernel immediately before the call on the stream.
 * Otherwise as splitk_gemm_bf16().
 */
SPLITK_API int splitk_gemm_bf16_bias(const void *a, const void *b, const void *bias,
                                     void *c, int M, int N, int K, int L,
                                     int split_k, splitk_stream_t stream);

/*
 * As splitk_gemm_bf16() with an explicit plan (from splitk_plan() or
 * splitk_plan_for(), possibly with stages / mailbox fields edited; the call
 * re-validates it) and flags (SPLITK_FLAG_NO_PDL).
 */
SPLITK_API int splitk_gemm_bf16_planned(const void *a, const void *b, void *c,
                                        int M, int N, int K, int L,
                                        const splitk_plan_t *plan,
                                        unsigned flags, splitk_stream_t stream);

/*
 * End-to-end call with host activations and host output: enqueues on
 * `stream` the copy b_host -> b_dev (M*K*L bf16), the GEMM with the resident
 * device weights `a`, and the copy c_dev -> c_host (M*N*L bf16).  b_dev and
 * c_dev are caller-owned device buffers of those sizes.  When both host
 * buffers are page-locked and mapped into the device address space (and all
 * four buffers 16-byte aligned), the two copies are small kernels chained to
 * the GEMM by programmatic dependent launch: the GEMM is resident and streams
 * its weights while the activations arrive, and every copy still waits for
 * the work ahead of it in the stream before touching memory.  Otherwise the
 * copy engines do them (pageable host memory: not asynchronous).  The
 * caller synchronizes `stream` before reading c_host.
 */
SPLITK_API int splitk_gemm_bf16_hostio(const void *a, const void *b_host,
                                       void *c_host, void *b_dev, void *c_dev,
                                       int M, int N, int K, int L, int split_k,
                                       splitk_stream_t stream);

/*
 * End-to-end call without copy engines: the GEMM reads the activations
 * straight from pinned host memory `b_host` (B[L][M][K] bf16) and writes C
 * straight into pinned host memory `c_host` (C[L][M][N] bf16), both through
 * their device mappings (on a coherent CPU-GPU link, the epilogue threads'
 * loads and stores cross it within the kernel).  Both buffers must be
 * page-locked and mapped into the device address space (cudaHostAlloc /
 * cudaMallocHost, or registered with cudaHostRegister and the mapped flag):
 * otherwise SPLITK_ERR_NOT_MAPPED, with nothing enqueued.  Only plans whose
 * activations the epilogue threads load (the staged decode tactic: narrow
 * tiles, short K slices) can do this; other shapes return
 * SPLITK_ERR_NO_FIT (use splitk_gemm_bf16_hostio).  The caller synchronizes
 * `stream` before reading c_host and keeps b_host unchanged until then.
 */
SPLITK_API int splitk_gemm_bf16_zerocopy(const void *a, const void *b_host, void *c_host,
                                         int M, int N, int K, int L, int split_k,
                                         splitk_stream_t stream);

/*
 * splitk_gemm_bf16() for callers that must not allocate device memory.
 * (No counterpart on the method's pages; this is a library entry point.)
 *
 * Who needs it: code that runs where cudaMalloc is not an option -- inside a
 * framework whose caching allocator owns the device memory budget, on a
 * latency-critical path where cudaMalloc's implicit synchronisation and
 * global lock are unacceptable, or in a process that pre-reserves all GPU
 * memory and treats any later allocation as a failure.  splitk_gemm_bf16()
 * allocates its tensor-map pool (and a pinned host mirror) on its first call;
 * this entry point allocates nothing: no cudaMalloc, cudaFree or allocating
 * library routine, and no host-side cache.
 *
 * Arguments, layouts, tiling and results are those of splitk_gemm_bf16()
 * (same kernel, same plan; outputs are bit-identical).  The only scratch the
 * kernel reads besides A, B and C -- one 128-byte CUDA tensor map of A -- is
 * kept in a file-scope device array of 256 bytes inside the library, which
 * every GPU that loads the library holds until the process exits.  A call
 * whose scratch would exceed that array is rejected with SPLITK_ERR_SCRATCH
 * (with one 128-byte map per call, no valid call does).
 *
 * The first call on a device (with that device current) looks up the
 * array's device address once (cudaGetSymbolAddress).  Every call rewrites
 * the whole map on `stream` with a host-to-device copy ahead of its kernel,
 * so nothing in the array has to start at zero and the array keeps the last
 * call's map.  That copy reads a host buffer that lives only during the
 * call, so a call on a stream that is capturing a CUDA graph is refused
 * with SPLITK_ERR_CAPTURE, with nothing enqueued (a captured copy would
 * read that buffer again at every replay).  All calls
 * on a device share that one array (each device has its own copy): calls
 * that overlap on the GPU, such as calls on two streams of one device,
 * race on it.  Calls issued in order on one stream do not overlap.
 *
 * The array's device address is looked up once per device and kept for the
 * life of the process (as are the plan's device properties): a
 * cudaDeviceReset() after the first call on a device is not supported.
 */
SPLITK_API int splitk_gemm_bf16_noalloc(const void *a, const void *b, void *c,
                                        int M, int N, int K, int L, int split_k,
                                        splitk_stream_t stream);

/*
 * Diagnostic record of the first bounded wait that ran out on the current
 * device since the last read (the Muse Spark AMD dev page's _spin_bounded:
 * every wait is bounded, the first timeout leaves a record and a sticky
 * failed state, later waits of the launch give up at once).
 */
typedef struct splitk_fault_t {
    int code;        /* SPLITK_OK or SPLITK_ERR_TIMEOUT                        */
    int role;        /* 0 weight TMA, 1 activation TMA, 2 MMA, 3 TMEM release,
                        4 epilogue: MMA completion, 5 epilogue: partials
                        (rank 0), 6 epilogue: mailbox free (peer), 7 A16W4
                        decode, 8 MMA: accumulator free (persistent plans)   */
    int index;       /* K tile or reduction round being waited for             */
    int parity;      /* mbarrier phase parity waited for                       */
    int block[3];    /* blockIdx of the CTA                                    */
    int cluster_rank;
} splitk_fault_t;

/*
 * Synchronizes the current device, copies its fault record into *out (when
 * out is not NULL), clears it, and returns its code (SPLITK_OK when no wait
 * ran out, SPLITK_ERR_TIMEOUT otherwise, SPLITK_ERR_CUDA if the device
 * cannot be read).
 */
SPLITK_API int splitk_get_fault(splitk_fault_t *out);

/* splitk_get_fault(NULL). */
SPLITK_API int splitk_get_status(void);

/*
 * Upper bound, in nanoseconds of %globaltimer, of every wait inside the
 * kernel for launches made after this call (default 1e9 = 1 s).  ns = 0
 * restores the default.
 */
SPLITK_API int splitk_set_wait_limit_ns(uint64_t ns);

/*
 * Test-only fault injection for launches made after this call.
 * SPLITK_INJECT_SKIP_PUBLISH: cluster ranks other than 0 skip publishing
 * their partials, so rank 0's bounded wait for them runs out and the call
 * reports SPLITK_ERR_TIMEOUT (the output is then undefined).  No GPU fault is
 * involved: nothing is stored remotely and every wait stays bounded.
 * 0 turns injection off.
 */
#define SPLITK_INJECT_SKIP_PUBLISH 0x1u
SPLITK_API int splitk_debug_inject(unsigned flags);

/*
 * Timeline tracing for launches made after this call.  `device_buffer`
 * (caller-owned device memory, 8-byte aligned) receives, for each CTA with
 * linear index (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x
 * below bytes / 128, sixteen uint64 words: [0] SM id | cluster rank << 32,
 * then %globaltimer nanoseconds at [1] CTA start, [2] set-up barrier passed,
 * [3] last weight TMA issued, [4] activation producer past the PDL wait,
 * [5] first and [6] last ring stage landed (MMA issuer), [7] accumulator
 * complete, [8] partials published (ranks != 0) or summed (rank 0),
 * [9] tile stored (rank 0), [10] CTA end, [11] mbarriers initialised,
 * [12] A's tensor map acquired, [13] first ring pass of weight loads issued,
 * [14] TMEM allocated, [15] epilogue past the set-up barrier.  Words never
 * reached stay as they were.  NULL (or bytes = 0) turns tracing off.
 */
SPLITK_API int splitk_set_trace(void *device_buffer, size_t bytes);

/*
 * The memory the library owns on the current device (no counterpart on the
 * method's pages; a library accounting call): *device_bytes of device memory
 * (the tensor-map pool of A, 0 until the first call that needs it),
 * *host_bytes of page-locked host memory (the pool's mirror) and *maps
 * tensor maps of A in the pool.  Any of the pointers may be NULL.  Reads the
 * library's own bookkeeping only: no allocation, no synchronisation, and no
 * CUDA call but the lookup of the current device
 * (SPLITK_ERR_UNSUPPORTED_DEVICE if there is none).
 */
SPLITK_API int splitk_cache_info(size_t *device_bytes, size_t *host_bytes, int *maps);

/* Synchronizes every device the library used, then frees its caches.  A
 * CUDA graph that captured calls of this library holds addresses of the freed
 * tensor maps: do not replay it after this call (capture it again). */
SPLITK_API void splitk_release(void);

/* A static description of a status code. */
SPLITK_API const char *splitk_strerror(int code);

/* Library version: major * 10000 + minor * 100 + patch. */
SPLITK_API int splitk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPLITK_H */
