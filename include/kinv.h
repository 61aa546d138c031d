/*
 * kinv.h -- C ABI of libkinv, a batch-invariant LLM forward step for NVIDIA
 * GB300 (sm_103a).
 *
 * What "batch-invariant" means here ("Deterministic and bit-exact inference",
 * trustbutveri.fyi record M-0002, *technical* and *How it works*): every
 * kernel fixes the reduction order of each output element whatever the batch
 * size, so the bits of row i (request b) depend only on row i's own inputs --
 * not on how many rows share the call, which rows they are, where row i sits
 * in the batch, or how a prompt was chunked.  The three reductions the pages
 * name are RMSNorm, matrix multiplication and attention; attention splits the
 * key/value dimension by a FIXED SPLIT SIZE, not a fixed number of splits.
 * The promise holds within one device class and one build (Kinetic
 * "Receipts", *What a receipt proves*: bits are promised only within one class
 * and one build); kinv_device_class() and kinv_build_id() name both.
 *
 * Conventions for every call below:
 *  - Pointers marked "device" are CUDA device pointers owned by the caller.
 *    The library never allocates, frees or synchronises on these paths; each
 *    call enqueues its kernels on `stream` (NULL = the legacy default stream)
 *    and returns.  Scratch space is passed in by the caller (`workspace`,
 *    sized by the matching *_workspace() query).
 *  - bf16 tensors are IEEE bfloat16 bit patterns, row-major, with the leading
 *    dimension (`ld*`, in elements) given.  fp32 accumulation throughout.
 *  - Errors are returned, never thrown, and nothing is launched when a call
 *    returns an error.  Shape, alignment and workspace checks happen on the
 *    host before any launch.  Launch failures return KINV_ERR_CUDA.  A device
 *    wait that runs out of time (every spin in the kernels is bounded) records
 *    a code in a device status word that kinv_last_device_status() reports.
 *  - Calls are thread-safe; the only global state is a lock-guarded cache,
 *    per CUDA context, of device attributes, of the device address of the
 *    status word and of kernel shared-memory limits.
 */
#ifndef KINV_H
#define KINV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* kinv_stream; /* same type as cudaStream_t */

typedef enum {
  KINV_OK = 0,
  KINV_ERR_INVALID_ARG = -1, /* null pointer, negative size, bad enum */
  KINV_ERR_UNSUPPORTED = -2, /* a shape or setting outside the supported set */
  KINV_ERR_ALIGNMENT = -3,   /* base or leading dimension not 16-byte aligned */
  KINV_ERR_WORKSPACE = -4,   /* workspace missing or smaller than the query */
  KINV_ERR_CUDA = -5,        /* a CUDA runtime/driver call failed */
  KINV_ERR_TIMEOUT = -6      /* a bounded device-side wait gave up */
} kinv_status;

typedef enum { KINV_BF16 = 0, KINV_F32 = 1 } kinv_dtype;

/* Human-readable name of a status code (static string). */
const char* kinv_status_string(int status);

/* Device class whose bits this build promises: "cuda-sm103a". */
const char* kinv_device_class(void);

/* Build id: 16 hex digits identifying this build of the kernels (a hash of
 * the sources and compile flags, fixed at build time).  Kinetic "Receipts",
 * *Making a receipt*: the receipt's build field pins every compiled kernel. */
const char* kinv_build_id(void);

/* Synchronises `stream`, then returns and clears the device status word of the
 * current device: KINV_OK, or the last code recorded since the previous call --
 * KINV_ERR_TIMEOUT (a bounded wait gave up), KINV_ERR_INVALID_ARG (an
 * attention call met a device-side length outside its stated bounds) or
 * KINV_ERR_UNSUPPORTED (a sampler row outside the supported settings).
 * Returns KINV_ERR_CUDA if the synchronisation itself fails. */
int kinv_last_device_status(kinv_stream stream);

/* Self-test of the bounded device waits (no counterpart on the pages; the
 * failure-detection rule every kernel here follows): launches one thread
 * block that waits on a shared-memory barrier nothing ever completes, for at
 * most limit_ns nanoseconds (1000 <= limit_ns <= 100000000), with the same
 * bounded-wait code the GEMM's pipeline waits use.  The wait gives up, records
 * KINV_ERR_TIMEOUT in the status word and the block exits, so the next
 * kinv_last_device_status() returns KINV_ERR_TIMEOUT and the context stays
 * usable.  Errors: KINV_ERR_INVALID_ARG for a limit outside the range. */
kinv_status kinv_test_bounded_wait(int64_t limit_ns, kinv_stream stream);

/* ------------------------------------------------------------------ GEMM
 * C[M][N] = A[M][K] . W[N][K]^T   ("Deterministic and bit-exact inference",
 * *technical*: batch-invariant matrix multiplication).
 *
 * A, W: device bf16, row-major, leading dimensions lda, ldw (elements).
 * C: device, bf16 (c_dtype = KINV_BF16) or fp32 (KINV_F32), leading dim ldc.
 * Arithmetic: bf16 products, fp32 accumulation on the tensor cores, one
 * rounding at the store.  The tile shape, the K order (ascending blocks of 64)
 * and the constant split of K (summed in fixed rank order) are chosen from
 * (N, K) alone, never from M: row i's bits are the same for every M.
 * Requirements: K % 64 == 0, N % 16 == 0, M >= 0; A, W, C 16-byte aligned;
 * lda, ldw multiples of 8; ldc a multiple of 8 (bf16) or 4 (fp32).
 * Errors: KINV_ERR_UNSUPPORTED / KINV_ERR_ALIGNMENT / KINV_ERR_INVALID_ARG.
 * M == 0 returns KINV_OK and launches nothing. */
kinv_status kinv_gemm(const void* A, int64_t lda, const void* W, int64_t ldw,
                      void* C, int64_t ldc, kinv_dtype c_dtype,
                      int M, int N, int K, kinv_stream stream);

/* RMSNorm folded into the projections around it ("Deterministic and
 * bit-exact inference", *technical*: batch-invariant RMSNorm and matmul).
 * The RMSNorm of a residual-stream row x, h = x / rms(x) * g, feeds only a
 * projection h . W^T, which equals (x . (W * g)^T) / rms(x) with the gain g
 * folded into W's columns once.  So:
 *  - a producing projection (`resid`) adds its bf16 output to the residual
 *    stream in its epilogue, resid[m][n] = bf16(resid[m][n] + out) with out
 *    the fp32 product (one rounding: the projection's output is not stored),
 *    and leaves the new row's sum of squares over each 128-column tile in
 *    ss_out[m][n / 128] (no other output; C may be NULL);
 *  - a consuming projection (`row_ss`) multiplies its fp32 result row m by
 *    1 / sqrt((row_ss[m][0] + row_ss[m][1] + ...) / norm_dim + eps), the
 *    tiles added in ascending order, before its rounding or epilogue;
 * so h is never rounded or stored.  Each partial and each row's total is
 * formed in a fixed order, so the bits do not depend on the batch.
 * row_ss: device fp32 [M][row_ss_tiles]; resid: device bf16 [M][N] (ld_resid,
 * a multiple of 8, N % 128 == 0); ss_out: device fp32 [M][N / 128]. */
typedef struct {
  const float* row_ss;
  int row_ss_tiles;
  int norm_dim;
  float eps;
  void* resid;
  int64_t ld_resid;
  float* ss_out;
} kinv_gemm_fusion;

/* kinv_gemm with the folded-RMSNorm options above (fusion nullable: plain
 * kinv_gemm).  Same tile, K order and split as kinv_gemm. */
kinv_status kinv_gemm_fused(const void* A, int64_t lda, const void* W, int64_t ldw,
                            void* C, int64_t ldc, kinv_dtype c_dtype, int M, int N, int K,
                            const kinv_gemm_fusion* fusion, kinv_stream stream);

/* Partial sums of squares of bf16 rows for a consuming projection's folded
 * RMSNorm (the first layer, whose input comes from the embedding):
 * ss_out[r][t] = sum over the 128 columns c of tile t of x[r][c]^2, in column
 * order.  x: device bf16 [rows][dim] (ldx); dim % 128 == 0. */
kinv_status kinv_row_sumsq(const void* x, int64_t ldx, int rows, int dim, float* ss_out,
                           kinv_stream stream);

/* QKV projection with kinv_rope_append in the epilogue: the product
 * qkv = A . W_qkv^T is formed with the same tile, K order and split as
 * kinv_gemm (N = (Hq + 2 Hkv) D), rounded to bf16 as kinv_gemm would store it,
 * and then, without going through memory, handled exactly as kinv_rope_append
 * handles its qkv rows (the same per-head arithmetic): q heads -> q_out, k heads
 * (RoPE, optional QK-norm) and v heads -> the caches at (seq[m], pos[m]).  The
 * result is bit-identical to kinv_gemm followed by kinv_rope_append
 * ("Deterministic and bit-exact inference", *technical*: the matmul is one of
 * the batch-invariant kernels; RoPE and the append reduce nothing across rows).
 * A bf16 [M][K] (lda), W_qkv bf16 [N][K] (ldw); q_out bf16 [M][Hq][D]; caches,
 * strides, seq, pos, norms, eps and rope_base as in kinv_rope_append.
 * fusion (nullable): the folded input RMSNorm (row_ss) of kinv_gemm_fused;
 * `resid` is not allowed here.
 * Requirements: D in {64, 128}, N % 128 == 0, K % 64 == 0, 16-byte alignment. */
kinv_status kinv_gemm_qkv_rope(const void* A, int64_t lda, const void* W_qkv, int64_t ldw,
                               void* q_out, void* k_cache, void* v_cache, int64_t seq_stride,
                               int64_t tok_stride, const int32_t* seq, const int32_t* pos,
                               const void* q_norm, const void* k_norm, float eps, int M, int Hq,
                               int Hkv, int D, int K, float rope_base,
                               const kinv_gemm_fusion* fusion, kinv_stream stream);

/* Gate/up projection with the SwiGLU applied in the epilogue:
 *   act[m][f] = bf16(silu(g) * u),  silu(g) = g / (1 + e^-g),
 *   g = A[m] . Wgate[f],  u = A[m] . Wup[f]  (fp32 accumulators, never rounded)
 * with the same tile, K order and split as kinv_gemm for N = 2F (so a row's
 * bits do not depend on M).  W_gu holds the 2F weight rows interleaved in
 * blocks of 64: rows 128j .. 128j+63 are gate rows 64j .. 64j+63 and rows
 * 128j+64 .. 128j+127 are up rows 64j .. 64j+63.  act: bf16 [M][F], leading
 * dimension ld_act (a multiple of 8).  fusion (nullable): the folded input
 * RMSNorm (row_ss) of kinv_gemm_fused, applied to g and u; `resid` is not
 * allowed here.  Requirements: F % 64 == 0, K % 64 == 0, alignment as for
 * kinv_gemm. */
kinv_status kinv_gemm_swiglu(const void* A, int64_t lda, const void* W_gu, int64_t ldw,
                             void* act, int64_t ld_act, int M, int F, int K,
                             const kinv_gemm_fusion* fusion, kinv_stream stream);

/* --------------------------------------------------------------- RMSNorm
 * y[r][i] = x[r][i] / sqrt(mean_j x[r][j]^2 + eps) * w[i]
 * ("Deterministic and bit-exact inference", *technical*: batch-invariant
 * RMSNorm).  One thread block per row, its size a function of `dim`; each
 * thread sums the squares of its chunks in a fixed order, a fixed xor
 * butterfly adds the lanes of a warp, and the warp sums are added in
 * ascending order, so a row's bits do not depend on `rows`.
 * residual (nullable): when given, s = bf16(x + residual) is formed first,
 * written back into `x` (the new residual stream), and y = RMSNorm(s).
 * x, residual, y: device bf16 [rows][dim] with leading dims ldx, ldx, ldy.
 * w: device bf16 [dim].  Requirements: dim % 8 == 0, 8 <= dim <= 16384,
 * 16-byte aligned bases, ldx and ldy multiples of 8.  `x` may be const when
 * residual is NULL (it is not written). */
kinv_status kinv_rmsnorm(void* x, int64_t ldx, const void* residual,
                         const void* w, void* y, int64_t ldy,
                         int rows, int dim, float eps, kinv_stream stream);

/* ------------------------------------------------------ decode attention
 * out[b][h] = sum_{j < L_b} softmax_j(scale * q[b][h] . k[b][j][g]) v[b][j][g],
 * g = h / (Hq / Hkv)  ("Deterministic and bit-exact inference", *technical*:
 * attention is batch-invariant when the keys are cut into splits of one fixed
 * length, whatever their number).
 *
 * Keys of sequence b are cut into splits of `split_len` keys at absolute
 * offsets 0, split_len, 2 split_len, ...; each split yields an fp32 partial
 * (max, sum of exponentials, unnormalised output) and the partials are folded
 * in ascending split order.  The cut depends only on L_b, so a sequence's bits
 * do not depend on its batch-mates or their lengths.  L_b == 0 gives zeros.
 * Within a split the softmax is taken in base 2: with r = q . k (fp32) and
 * c = fp32(scale * log2 e), m = fp32(max r * c) and the weights
 * e = 2^fma(r, c, -m) (the hardware's approximate exp2) are formed in fp32,
 * summed in fp32, and enter the tensor cores as the bf16 pair hi = bf16(e),
 * lo = bf16(e - hi), so they keep about 16 significant bits; P.V is one fp32
 * chain over 16-key steps, each adding its hi . V, then its lo . V.
 *
 * q, out: device bf16 [B][Hq][D] (contiguous).  k_cache, v_cache: device bf16;
 *   element (b, j, g, d) is at b*seq_stride + j*tok_stride + g*D + d
 *   (elements); e.g. a contiguous [B][Lmax][Hkv][D] cache has
 *   seq_stride = Lmax*Hkv*D, tok_stride = Hkv*D.
 * kv_len: device int32 [B], each in [0, Lmax]; a sequence whose kv_len lies
 *   outside gets zeros, and the status word records KINV_ERR_INVALID_ARG
 *   (no key beyond Lmax is read).
 * workspace: device, at least kinv_attn_decode_workspace(B, Hq, D, Lmax,
 *   split_len) bytes, 16-byte aligned.
 * Requirements: D in {64, 128}; Hq % Hkv == 0; Hq / Hkv in {1, 2, 4, 8};
 * split_len == 256; strides multiples of 8.  A scale that is not a positive
 * finite number means 1/sqrt(D). */
size_t kinv_attn_decode_workspace(int B, int Hq, int D, int Lmax, int split_len);
kinv_status kinv_attn_decode(const void* q, const void* k_cache, const void* v_cache,
                             int64_t seq_stride, int64_t tok_stride,
                             const int32_t* kv_len, void* out,
                             int B, int Hq, int Hkv, int D, int Lmax, int split_len,
                             float scale, void* workspace, size_t workspace_bytes,
                             kinv_stream stream);

/* --------------------------------------- decode attention, no allocation
 * The pages have no counterpart to this call: it exists for callers that
 * cannot allocate device memory.  Some code cannot call cudaMalloc -- a plug-in
 * whose host program owns every byte of device memory through its own pool, a
 * real-time loop that must not take the allocator's implicit device-wide
 * synchronisation, or a binding with no device allocator at all -- and so
 * cannot provide the scratch that kinv_attn_decode takes as `workspace`.
 *
 * Same arguments, arithmetic and output bits as kinv_attn_decode, minus the
 * workspace: the split partials live in a scratch array compiled into the
 * library (KINV_NOALLOC_SCRATCH_BYTES bytes on every GPU that loads it, held
 * until the process exits).  Nothing is allocated or freed.
 *  - A call whose partials need more than KINV_NOALLOC_SCRATCH_BYTES (that is,
 *    kinv_attn_decode_workspace(B, Hq, D, Lmax, split_len) is larger) returns
 *    KINV_ERR_WORKSPACE and launches nothing.
 *  - The first call in each CUDA context (normally once per device) looks up
 *    the array's device address with that device current, checks the lookup
 *    and caches the address for that context; make that first call before any
 *    stream capture.
 *  - Every call on a device shares the one array, which keeps whatever the
 *    last call left in it (each call writes every partial it later reads, so
 *    nothing needs clearing).  Calls that overlap on the GPU -- on two streams,
 *    or from two threads -- race on it: serialise them. */
#define KINV_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
kinv_status kinv_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                     int64_t seq_stride, int64_t tok_stride,
                                     const int32_t* kv_len, void* out,
                                     int B, int Hq, int Hkv, int D, int Lmax, int split_len,
                                     float scale, kinv_stream stream);

/* ----------------------------------------------------- prefill attention
 * Causal attention for chunks of new query rows against the cache (which
 * must already hold their keys).  Sequence b contributes q_len[b] rows,
 * stored at rows q_offset[b] .. q_offset[b] + q_len[b] - 1 of q/out, at
 * absolute positions q_start[b] .. q_start[b] + q_len[b] - 1; the row at
 * position p attends to keys 0..p of sequence b.
 * Each row is computed with exactly the arithmetic of kinv_attn_decode for a
 * sequence of length p + 1 (same splits at absolute offsets, same fold), so a
 * row's bits do not depend on the chunking, on p0, on the other rows, and a
 * decode step equals a one-row prefill bit for bit.
 * The rows run on the tcgen05 tensor cores, 128 (row, head) pairs of one
 * sequence and kv head per thread block, which folds the sequence's splits
 * one after another in registers: kinv_attn_prefill_workspace() is 0 and
 * `workspace` may be NULL.
 * q, out: device bf16 [total_rows][Hq][D].  q_start, q_len, q_offset: device
 * int32 [B].  Caches and strides as for decode, the cache holding at least
 * max_kv keys of each of the B sequences (seq_stride > 0 when B > 1).  max_q_len bounds q_len[b],
 * max_kv bounds q_start[b] + q_len[b] (both used to size the grid and the
 * workspace), and q_offset[b] + q_len[b] <= total_rows; a sequence whose
 * device-side values break one of these bounds (or is negative) is left out
 * -- its rows of `out` are not written -- and the status word records
 * KINV_ERR_INVALID_ARG.  Requirements as for decode. */
size_t kinv_attn_prefill_workspace(int total_rows, int Hq, int D, int max_kv, int split_len);
kinv_status kinv_attn_prefill(const void* q, const void* k_cache, const void* v_cache,
                              int64_t seq_stride, int64_t tok_stride,
                              const int32_t* q_start, const int32_t* q_len,
                              const int32_t* q_offset, void* out,
                              int B, int total_rows, int max_q_len, int max_kv,
                              int Hq, int Hkv, int D, int split_len, float scale,
                              void* workspace, size_t workspace_bytes,
                              kinv_stream stream);

/* --------------------------------------------------------------- sampler
 * Seeded sampler with the settings a Kinetic receipt records (Kinetic
 * "Receipts", *Making a receipt*, the `sampling` object).  Per row b, in this
 * order: the logit bias (each entry (id, bias) of the row's list adds bias to
 * logit id in fp32, in list order; ids outside [0, V) are ignored); the
 * penalties over the distinct ids among the last repeat_last_n
 * history tokens (n < 0: all, n == 0: none), first the repeat penalty
 * (z/r if z > 0 else z*r), then, when presence_penalty or frequency_penalty is
 * not 0, z - (c * frequency_penalty + presence_penalty) with c the id's count
 * in that window (each operation rounded to fp32);
 * temperature <= 0 -> greedy argmax (lowest id on ties); otherwise the top_k
 * candidates ordered by (z desc, id asc); s = z / temperature;
 * e_i = exp(s_i - s_0); typical-p (when 0 < typical_p < 1) keeps, with
 * p_i = e_i / sum(e) and H = -sum p_i log p_i, the shortest set of candidates
 * taken by |-log p_i - H| ascending (then candidate order) whose p reaches
 * typical_p, and the steps below see only that set, in candidate order;
 * top-p keeps the shortest prefix whose sum of e reaches top_p * sum(e)
 * (skipped when top_p >= 1); min-p keeps e_i >= min_p * e_first, e_first the
 * first kept candidate's e (skipped when min_p <= 0); then u = (Philox4x32-10(counter = (step lo, step hi, 0, 0),
 * key = (seed lo, seed hi)).word0 >> 8) * 2^-24 picks the first kept candidate
 * whose running sum of e exceeds u * (sum of kept e).  The counter is the
 * request's own step, never its batch slot: the drawn token depends only on
 * the row's logits, history, settings and step.  A cluster of up to eight
 * thread blocks shares a row (the count follows the batch size; the token
 * does not depend on it); ranking and thresholds are compare-only on fp32
 * values; sums in fixed order.
 * top_k <= 0 (or >= V) means the whole vocabulary: e is then summed over all
 * V ids (per 128-id block, blocks in order) and the top-p / min-p cut must
 * fall within the 1024 most likely ids.
 *
 * logits: device fp32 [B][ld]; params: device kinv_sampling_params [B];
 * history: device int32 [B][hist_ld], row b holding hist_len[b] ids, oldest
 * first; step: device int64 [B]; out_tokens: device int32 [B].
 * Requirements: 1 <= V; ld >= V; top_k in [1, 1024] or the whole vocabulary
 * (V <= 262144, and top_p < 1 or min_p > 0 cutting within the 1024 most
 * likely ids, typical-p off) unless temperature <= 0; hist_len[b] <= hist_ld <= 1024
 * (else KINV_ERR_UNSUPPORTED before launch); at most 1024 logit-bias entries
 * per row (further entries are ignored).  Rows whose
 * settings or logits fall outside this set get token -1 and the device status
 * word records KINV_ERR_UNSUPPORTED. */
typedef struct {
  int32_t id;
  float bias;
} kinv_logit_bias;

typedef struct {
  float temperature;
  float top_p;
  float min_p;
  float repeat_penalty;
  int32_t top_k;
  int32_t repeat_last_n;
  uint64_t seed;
  float presence_penalty;   /* 0: off */
  float frequency_penalty;  /* 0: off */
  const kinv_logit_bias* logit_bias;  /* device, n_logit_bias entries; NULL: none */
  int32_t n_logit_bias;               /* at most 1024 */
  float typical_p;                    /* on when 0 < typical_p < 1 */
} kinv_sampling_params;

size_t kinv_sample_workspace(int B, int V);
kinv_status kinv_sample(const float* logits, int64_t ld, int B, int V,
                        const kinv_sampling_params* params,
                        const int32_t* history, int hist_ld, const int32_t* hist_len,
                        const int64_t* step, int32_t* out_tokens,
                        void* workspace, size_t workspace_bytes, kinv_stream stream);

/* ------------------------------------------------------------ layer glue
 * Element-wise steps of the decoder block.  None of them sums across
 * elements, so each is batch-invariant by construction. */

/* out[r] = table[ids[r]] for r < rows; table bf16 [vocab][dim] (ld = dim),
 * ids device int32 [rows] (ids outside [0, vocab) give zeros), dim % 8 == 0. */
kinv_status kinv_embed(const void* table, int vocab, int dim, const int32_t* ids,
                       void* out, int rows, kinv_stream stream);

/* out[n][k] = bf16(w[n][k] * g[k]) (fp32 product): an RMSNorm gain g moved
 * into the input columns of the projection it feeds, once, when the weights are
 * loaded ("Deterministic and bit-exact inference", *technical*: RMSNorm and
 * matmul; see kinv_gemm_fusion).  w, out: device bf16 [N][K] (ldw, ldo
 * multiples of 8; out may equal w); g: device bf16 [K]; K % 8 == 0,
 * N <= 262140, 16-byte aligned bases. */
kinv_status kinv_scale_columns(const void* w, int64_t ldw, const void* g, void* out, int64_t ldo,
                               int N, int K, kinv_stream stream);

/* out = bf16(x + y), n elements, bf16, n % 8 == 0, 16-byte aligned. */
kinv_status kinv_add(const void* x, const void* y, void* out, int64_t n, kinv_stream stream);

/* out[r][i] = bf16(silu(gu[r][i]) * gu[r][F + i]), silu(g) = g / (1 + e^-g);
 * gu bf16 [rows][2F] (ld_gu), out bf16 [rows][F] (ld_out); F % 8 == 0. */
kinv_status kinv_swiglu(const void* gu, int64_t ld_gu, void* out, int64_t ld_out,
                        int rows, int F, kinv_stream stream);

/* Rotary embedding (rotate-half pairs (i, i + D/2), theta_i = p * base^(-2i/D))
 * with optional per-head RMSNorm first (q_norm / k_norm nullable, gains [D]),
 * then the key/value append: for row r of sequence seq[r] at absolute position
 * pos[r]:
 *   q_out[r][h]                = bf16(RoPE(norm(q)))        h < Hq
 *   k_cache[seq][pos][g]       = bf16(RoPE(norm(k)))        g < Hkv
 *   v_cache[seq][pos][g]       = v                           (copied bits)
 * qkv: device bf16 [rows][(Hq + 2 Hkv) D] (ld_qkv), q, k, v heads in that
 * order.  q_out: bf16 [rows][Hq][D].  seq, pos: device int32 [rows].
 * Requirements: D in {64, 128}; strides multiples of 8; 16-byte alignment. */
kinv_status kinv_rope_append(const void* qkv, int64_t ld_qkv, void* q_out,
                             void* k_cache, void* v_cache, int64_t seq_stride,
                             int64_t tok_stride, const int32_t* seq, const int32_t* pos,
                             const void* q_norm, const void* k_norm, float eps,
                             int rows, int Hq, int Hkv, int D, float rope_base,
                             kinv_stream stream);

/* One decode iteration's bookkeeping, per request b < B: append
 * tokens[b] to history row b (shifting out the oldest id once hist_len ==
 * hist_ld), hist_len[b] = min(hist_len[b] + 1, hist_ld), step[b] += 1, and
 * pos[b] += 1, kv_len[b] += 1 for whichever of pos / kv_len is not NULL.
 * All device pointers. */
kinv_status kinv_decode_advance(const int32_t* tokens, int32_t* history, int hist_ld,
                                int32_t* hist_len, int64_t* step, int32_t* pos,
                                int32_t* kv_len, int B, kinv_stream stream);

#ifdef __cplusplus
}
#endif
#endif /* KINV_H */
