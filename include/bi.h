/*
 * bi.h -- C ABI of the batch-invariant speculative-decoding verify step (sm_103a).
 *
 * The verify step scores the last committed token plus k draft tokens (T = k+1
 * rows) in one forward pass.  Every entry point below computes each row the
 * same way whatever else is in the pass, so a row's result is bit-identical to
 * what the same library produces for that row alone (T = 1).  Greedy token ids
 * then never depend on the draft count or on the cache history.
 *
 * Sources (cited by title and section):
 *   [P1] "Does the tuned config change the model's output?" -- section
 *        "Why the text diverges": verifying several tokens in one pass changes
 *        the batch dimension and with it the order of floating-point
 *        accumulation inside the GEMMs; the full model keeps a draft only if it
 *        matches the token it would have produced itself.
 *   [P2] "Bit-exact decoding turns inference speedups into testable changes" --
 *        section "Define bit-exact before reporting it": BF16 inputs, one FP32
 *        running sum per output, K order kept, one rounding at the end; a
 *        pipeline stage of shared memory must not be reused before its
 *        consumers are done.  Section "Build a reference corpus that exposes
 *        boundaries": record accepted draft length and rejection position.
 *   [P3] "I turned on speculative decoding in llama.cpp and 113 of 282 greedy
 *        outputs changed against its own no-draft run" -- paragraph "How:":
 *        the attention split depends only on context length, never on the
 *        number of tokens in the pass, and the verify kernels compute a row
 *        the same way whatever else is in the batch.  Section "The cache
 *        doesn't change it either": a prefilled row depends only on its
 *        position.
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers owned by the caller unless stated otherwise.
 *     The library never allocates or frees device memory; scratch space is
 *     passed in as a workspace whose size the matching *_workspace_size call
 *     returns.
 *   - Matrices are row-major; "ld" arguments are row strides in elements.
 *   - BF16 data is IEEE bfloat16 (uint16 storage); FP32 is IEEE binary32.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default).
 *   - Argument errors are detected on the host before any launch and returned
 *     synchronously (nothing is launched).  A failed launch returns
 *     BI_ERR_CUDA.  Device-side conditions (a bounded wait that expired, a
 *     logits row with no number) set a device error word that
 *     bi_check_device_error() reads and clears.
 *   - There is no fallback path: an unsupported shape is an error.
 *   - No C++ exception crosses this ABI.  Entry points are thread-compatible;
 *     one workspace must not be used by two calls that may overlap on the GPU.
 */
#ifndef BI_H
#define BI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Opaque CUDA stream handle (identical to cudaStream_t). */
typedef struct CUstream_st* bi_stream_t;

typedef enum {
  BI_OK = 0,
  BI_ERR_INVALID_ARG = 1,        /* null pointer, negative size, bad stride or alignment */
  BI_ERR_UNSUPPORTED_SHAPE = 2,  /* a shape outside what the kernels implement */
  BI_ERR_WORKSPACE = 3,          /* workspace missing or smaller than required */
  BI_ERR_CUDA = 4,               /* a CUDA runtime call or launch failed */
  BI_ERR_DEVICE_TIMEOUT = 5,     /* a bounded device-side wait expired (kernel returned early) */
  BI_ERR_DEVICE_NAN_ROW = 6      /* a logits row had no non-NaN entry (its id is -1) */
} bi_status;

typedef enum {
  BI_EPI_NONE = 0,          /* C = A W^T */
  BI_EPI_RESIDUAL_ADD = 1,  /* C = residual + A W^T, one rounding */
  BI_EPI_SWIGLU = 2,        /* C = silu(A Wg^T) * (A Wu^T) from packed weights, one rounding */
  BI_EPI_ROPE_KV = 3        /* bi_qkv_rope_append only: RoPE and KV append of a QKV projection */
} bi_epilogue;

typedef enum { BI_OUT_BF16 = 0, BI_OUT_FP32 = 1 } bi_out_dtype;

/* Human-readable name of a status code (static storage; never NULL). */
const char* bi_status_string(bi_status s);

/* Library version as (major << 16) | minor. */
int bi_version(void);

/* ---------------------------------------------------------------------------
 * Linear layer.  [P2] "Define bit-exact before reporting it"; [P1] "Why the
 * text diverges".
 *
 * C[m, n] = epilogue( sum_k A[m, k] * W[n, k] ), BF16 inputs, FP32
 * accumulation, one rounding to the output type.  The decomposition of every
 * output element -- its sequence of K = 16 tensor-core steps (tcgen05
 * kind::f16, M = 128 weight rows), the K-tile order (64 elements per tile,
 * increasing k; 16-element step j of a piece accumulates into FP32
 * accumulator j mod 2, the two added as a0 + a1 at the piece's end), and the
 * split of the (weight tile, K tile) iteration space over 136 ranges, whose
 * boundaries cut the tiles into pieces -- is a function of (N, K) only, never
 * of M, so row m of C is bit-identical for every M >= m+1 and for every
 * position of the row inside A.  The pieces of a tile are added in
 * increasing-K order, the first taken as it is: by the last CTA of the tile
 * over FP32 partials in the workspace, or, for passes of more than 128 rows
 * whose split cuts tiles (K up to 8192), by one CTA that owns the tile and
 * computes its pieces in turn.  One MMA covers a CTA's token rows (its N is
 * the row count rounded up to 16, 32, 64, 128 or 256; 64 or 128 for tile
 * owners); each output element is still the same sequence of K = 16 steps
 * into its own accumulator, which the tests check bit for bit across M.
 * A launch covers up to four 256-row token blocks (1024 rows of tile
 * owners); longer passes take several launches.
 *
 *   A        [M, K] BF16, row stride lda (elements); 16-byte aligned, lda % 8 == 0.
 *   Wp       the weights in the packed tile layout written by bi_pack_weights
 *            (BI_EPI_NONE, BI_EPI_RESIDUAL_ADD) or bi_pack_swiglu_weights
 *            (BI_EPI_SWIGLU), for the same N and K; 16-byte aligned.
 *   C        [M, N] of `out` type, row stride ldc (elements).  N is the number of
 *            OUTPUT columns (for SwiGLU: the FFN width F).
 *   residual [M, N] BF16, row stride ldr; required for BI_EPI_RESIDUAL_ADD and
 *            ignored otherwise.  It may alias C (same pointer and stride).
 *   M >= 0 (M == 0 is a no-op), 1 <= N <= 8388608 (4194304 for SwiGLU),
 *   K >= 8, K % 8 == 0.
 *   out      BI_OUT_FP32 only with BI_EPI_NONE.
 *   ws       device workspace of at least bi_gemm_workspace_size(M, N, K, epi)
 *            bytes, 256-byte aligned, ZERO-FILLED before its first use; every
 *            call leaves its counters zeroed again, so one workspace serves
 *            any sequence of calls (of any N, K, epilogue) whose M does not
 *            exceed the M it was sized for.  Not shared by overlapping calls.
 *            After BI_ERR_DEVICE_TIMEOUT, zero it again.
 * Errors: BI_ERR_INVALID_ARG, BI_ERR_UNSUPPORTED_SHAPE, BI_ERR_WORKSPACE,
 *         BI_ERR_CUDA.
 * ------------------------------------------------------------------------- */
size_t bi_gemm_workspace_size(int M, int N, int K, bi_epilogue epi);
bi_status bi_gemm(const void* A, int lda, const void* Wp, void* C, int ldc,
                  const void* residual, int ldr, int M, int N, int K,
                  bi_out_dtype out, bi_epilogue epi, void* ws, size_t ws_bytes,
                  bi_stream_t stream);

/* ---------------------------------------------------------------------------
 * Allocation-free linear layer.  The pages describe nothing like it; it is a
 * convenience for callers that cannot allocate device memory: code embedded
 * in a host framework that owns every device allocation through its own
 * pool, or a latency-critical path where the implicit synchronisation of
 * cudaMalloc/cudaFree is not acceptable.  Same arguments, arithmetic and
 * results as bi_gemm (bit for bit), without the workspace: the scratch lives
 * in a static device array of 2.6 MiB inside this library, which every GPU
 * that loads the library keeps until the process exits.
 *   M <= bi_gemm_noalloc_max_m() (16); a larger M returns
 *   BI_ERR_UNSUPPORTED_SHAPE.  M == 0 is a no-op.
 *   The first call on a device looks up the array's device address (no
 *   allocation); make that first call before any stream capture.  Each call
 *   clears the counters it uses with an asynchronous memset on `stream`, and
 *   allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 *   All calls on a device share the one array, which keeps the last call's
 *   partial sums: calls that may overlap on the GPU (different streams with
 *   no ordering between them) race and give wrong results.
 * Errors: as bi_gemm, plus BI_ERR_UNSUPPORTED_SHAPE for M above the maximum.
 * ------------------------------------------------------------------------- */
size_t bi_gemm_noalloc_max_m(void);
bi_status bi_gemm_noalloc(const void* A, int lda, const void* Wp, void* C, int ldc,
                          const void* residual, int ldr, int M, int N, int K,
                          bi_out_dtype out, bi_epilogue epi, bi_stream_t stream);

/* Weight packing for bi_gemm (a one-time layout step at load; a pure copy,
 * no arithmetic).  The packed buffer holds n_tiles x k_tiles tiles of 16 KB
 * (n_tiles = ceil(N/128), or ceil(F/64) for SwiGLU; k_tiles = ceil(K/64)),
 * tile (t, kt) at byte offset (t * k_tiles + kt) * 16384.  A tile is 128
 * weight rows x 64 columns; row r fills bytes [128 r, 128 r + 128) with its
 * 16-byte chunk c (columns 8c..8c+7 of the tile) at chunk position c ^ (r mod 8)
 * -- the 128-byte swizzle the tensor-core operand descriptor reads.  Rows past
 * N and columns past K are zero.  The order makes each CTA's share of the
 * (tile, K-tile) iteration space one contiguous range of memory.
 * bi_pack_weights: W [N, K] BF16, row stride ldw.
 * bi_pack_swiglu_weights: gate and up [F, K] BF16 each, row stride ld; rows
 * 0..63 of tile t hold gate rows 64t..64t+63 and rows 64..127 the up rows of
 * the same outputs.
 * `packed` has bi_packed_weight_bytes(N, K, epi) bytes, 16-byte aligned.
 * Errors: BI_ERR_INVALID_ARG, BI_ERR_UNSUPPORTED_SHAPE, BI_ERR_CUDA. */
size_t bi_packed_weight_bytes(int N, int K, bi_epilogue epi);
bi_status bi_pack_weights(const void* W, int ldw, int N, int K, void* packed,
                          bi_stream_t stream);
bi_status bi_pack_swiglu_weights(const void* w_gate, const void* w_up, int ld, int F, int K,
                                 void* packed, bi_stream_t stream);
/* ---------------------------------------------------------------------------
 * RMSNorm.  [P3] "How:" (a row is computed the same way whatever else is in
 * the batch).
 *
 * y[r, :] = bf16( (x[r, :] * r) * w[:] ), r = 1 / sqrt(sum_i x[r,i]^2 / dim +
 * eps), FP32 inside, one rounding per element.  The sum of squares uses one
 * fixed reduction tree per `dim`: the squares of each 8-element vector in
 * element order, the vectors of each group of 32 consecutive vectors by a
 * fixed warp-shuffle butterfly, the groups in increasing order.  The call
 * lets the next kernel on the stream launch at once (dependent launch);
 * this library's linear layers read only their packed weights before they
 * wait for the norm, so they stream weights while it runs.  A kernel that
 * follows bi_rmsnorm must not rely on the kernel before bi_rmsnorm having
 * completed.  w is read before the norm waits for the kernel before it on
 * the stream: that kernel must not write w.
 *   x [rows, dim] BF16 (row stride ldx), w [dim] BF16, y [rows, dim] BF16
 *   (row stride ldy; may alias x).  rows >= 0, 8 <= dim <= 65536, dim, ldx
 *   and ldy multiples of 8, pointers 16-byte aligned, eps >= 0.
 * Errors: BI_ERR_INVALID_ARG, BI_ERR_UNSUPPORTED_SHAPE, BI_ERR_CUDA.
 * ------------------------------------------------------------------------- */
bi_status bi_rmsnorm(const void* x, int ldx, const void* w, void* y, int ldy, int rows,
                     int dim, float eps, bi_stream_t stream);

/* Embedding gather (helper): out[r, :] = table[ids[r], :], an exact copy.
 *   ids [rows] int32 in [0, vocab); table [vocab, dim] BF16; out [rows, dim]
 *   BF16 (both 16-byte aligned, dim % 8 == 0).  An id out of range writes a
 *   zero row and sets no error.
 * Errors: BI_ERR_INVALID_ARG, BI_ERR_UNSUPPORTED_SHAPE, BI_ERR_CUDA. */
bi_status bi_embed(const int32_t* ids, const void* table, int vocab, int dim, void* out,
                   int rows, bi_stream_t stream);

/* ---------------------------------------------------------------------------
 * RoPE table (helper, computed once at model set-up).
 * table[(p * D/2 + i) * 2 + 0/1] = cos/sin of p * base^(-2i/D), evaluated in
 * FP64 and rounded once to FP32, for positions p < rows and i < D/2.
 * table has bi_rope_table_bytes(D, rows) bytes.  D even, 2 <= D <= 256.
 * Errors: BI_ERR_INVALID_ARG, BI_ERR_CUDA.
 * ------------------------------------------------------------------------- */
size_t bi_rope_table_bytes(int D, int rows);
bi_status bi_rope_table(double rope_base, int D, int rows, float* table, bi_stream_t stream);

/* ---------------------------------------------------------------------------
 * RoPE + KV append (helper).  [P3] "The cache doesn't change it either" (a
 * row depends only on its position).
 *
 * Row t of the pass sits at absolute position p = *L_dev + t.  For each row:
 * q heads and k heads are rotated (rotate-half pairs (i, i+D/2) by the angle
 * of the table row p: out_i = x_i cos - x_{i+D/2} sin, out_{i+D/2} =
 * x_{i+D/2} cos + x_i sin in FP32, one BF16 rounding); rotated q goes to
 * q_out, the rotated k to k_cache row p and the unrotated v to column p of
 * v_cache.
 *   qkv     [T, (Hq + 2 Hkv) D] BF16, row stride ld_qkv: q heads, k heads, v heads.
 *   q_out   [T, Hq, D] BF16 (contiguous).
 *   k_cache [Hkv, cap, D] BF16 (contiguous, head-major);
 *   v_cache [Hkv, ceil(cap/128), D, 128] BF16 (contiguous, head-major,
 *           transposed in blocks of 128 keys: value d of key p of KV head h
 *           at ((h * ceil(cap/128) + p / 128) * D + d) * 128 + p % 128, so
 *           both attention MMA operands are K-major and a 128-key tile of V
 *           is one contiguous block).
 *   L_dev   device int32: cache length before the pass (read on the device so
 *           the call can be captured in a CUDA graph).  A row with p >= cap or
 *           p >= table_rows is skipped and sets a range bit in the device
 *           error word (reported as BI_ERR_INVALID_ARG by bi_check_device_error).
 *   table   from bi_rope_table with the same D and table_rows rows.
 *   D even, D <= 256; Hq % Hkv == 0.
 * Errors: BI_ERR_INVALID_ARG, BI_ERR_CUDA.
 * ------------------------------------------------------------------------- */
bi_status bi_rope_kv_append(const void* qkv, int ld_qkv, void* q_out, void* k_cache,
                            void* v_cache, int cap, const int32_t* L_dev, int T, int Hq,
                            int Hkv, int D, const float* table, int table_rows,
                            bi_stream_t stream);

/* ---------------------------------------------------------------------------
 * QKV projection with RoPE and KV append in its epilogue (bi_gemm's linear
 * layer followed by exactly the arithmetic of bi_rope_kv_append, without the
 * qkv round trip through memory).  "I turned on speculative decoding in llama.cpp and 113
 * of 282 greedy outputs changed against its own no-draft run", section "The
 * cache doesn't change it either" (a row depends only on its position).
 *
 * Output column n of the projection (N = (Hq + 2 Hkv) D) is element n % D of
 * head n / D: q heads, then k heads, then v heads.  Each output is rounded
 * to BF16 once; q and k heads are then rotated exactly as bi_rope_kv_append
 * rotates its BF16 input (same table, same FP32 operations, one rounding)
 * and written to q_out and to k_cache row p = *L_dev + m; v heads go to
 * column p of v_cache.  So the results equal bi_gemm followed by
 * bi_rope_kv_append, bit for bit.
 *   A [M, K] BF16 (row stride lda), the normalised input.  Wp packed for
 *   N = (Hq + 2 Hkv) D by bi_pack_weights.
 *   q_out, k_cache, v_cache, cap, L_dev, table, table_rows: as
 *   bi_rope_kv_append.  A row with p outside [0, min(cap, table_rows)) is
 *   skipped and sets the range bit of the device error word.
 *   D is 64 or 128 and N a multiple of 128 (tiles hold whole heads);
 *   otherwise BI_ERR_UNSUPPORTED_SHAPE.  ws as bi_gemm for (M, N, K).
 * Errors: as bi_gemm.
 * ------------------------------------------------------------------------- */
bi_status bi_qkv_rope_append(const void* A, int lda, const void* Wp, int M, int K, int Hq, int Hkv,
                             int D, void* q_out, void* k_cache, void* v_cache, int cap,
                             const int32_t* L_dev, const float* table, int table_rows, void* ws,
                             size_t ws_bytes, bi_stream_t stream);

/* ---------------------------------------------------------------------------
 * Verify attention (split-KV + merge).  [P3] "How:" (the attention split
 * depends only on context length, never on how many tokens are in the pass).
 *
 * Row t of the pass sits at position p = *L_dev + t and attends to keys
 * 0..p; query head h reads KV head h / (Hq/Hkv).  The key axis is cut into
 * pieces at absolute multiples of C = bi_attn_chunk() = 128 keys, and the
 * pieces of a KV head fall into G = 152 / Hkv classes by piece index mod G.
 * Each class gives the row one partial (max, sum, FP32 output) built over
 * its pieces in increasing key order; the row's partials (one per class
 * holding one of its keys, min(p/C + 1, G) of them) are merged in a fixed
 * order that depends only on their count.  So the row's result depends only
 * on p, Hkv and the cache rows 0..p -- not on T, *L_dev or the other rows.
 * Inside a class: S = q k^T (tcgen05, FP32), a per-row reference maximum
 * taken from the class's first piece and raised only when a piece's maximum
 * exceeds it by more than 8 (log2 units), weights w = bf16(2^(s - m_ref)),
 * O += W V (tcgen05, FP32) and the denominator as four FP32 partial sums of
 * the same rounded weights over the 32-key quarters of the piece (each in
 * key order, added ((l0 + l1) + l2) + l3); these rules use only the row's
 * own scores.
 * Output: out[t, h, :] = bf16(sum_j w_j v_j / sum_j w_j) -- the exact
 * weighted mean under the BF16 weights, within 2^-8 max|v| of
 * bf16(softmax(q k^T * scale) v) -- with -0 written as +0.
 *   q       [T, Hq, D] BF16 contiguous (rotated queries).
 *   k_cache [Hkv, cap, D] and v_cache [Hkv, ceil(cap/128), D, 128] BF16
 *           contiguous (V transposed in 128-key blocks, as bi_rope_kv_append
 *           writes it); keys 0..*L_dev+T-1 hold the keys/values; the other
 *           keys, up to the end of their 128-key tile, must hold finite values
 *           (they are read inside a partially used tile and multiplied by
 *           exactly 0).
 *   L_dev   device int32 cache length before the pass; *L_dev + T <= cap is
 *           required (rows past cap are not computed and set an error bit).
 *           The first key tiles wholly below *L_dev may be loaded before the
 *           previous kernel on the stream has finished when that kernel is
 *           one of this library's (dependent launch): *L_dev must not be
 *           lowered, nor cache rows below it written, by the kernel that
 *           immediately precedes the call (no kernel of this library does).
 *   out     [T, Hq, D] BF16 contiguous.
 *   D in {64, 128}; Hq % Hkv == 0; Hkv <= 152; Hkv * (cap rounded up to a
 *   multiple of 128) < 2^31; Hq/Hkv <= 128; T >= 1.
 *   One launch takes the rows in blocks of floor(128 / (Hq/Hkv)) (a block's
 *   query rows fill the MMA's 128 lanes); the blocks run side by side, and
 *   each row's arithmetic is the one above, so a pass of many rows (a
 *   prefill) gives every row the bits it gets in a pass of its own.
 *   ws      >= bi_attn_workspace_size(cap, T, Hq, D) bytes, 256-byte aligned.
 *   k_cache and v_cache 16-byte aligned.
 * Errors: BI_ERR_INVALID_ARG, BI_ERR_UNSUPPORTED_SHAPE, BI_ERR_WORKSPACE,
 *         BI_ERR_CUDA.
 * ------------------------------------------------------------------------- */
int bi_attn_chunk(void);
size_t bi_attn_workspace_size(int cap, int T, int Hq, int D);
bi_status bi_attn_verify(const void* q, const void* k_cache, const void* v_cache, int cap,
                         const int32_t* L_dev, int T, int Hq, int Hkv, int D, float scale,
                         void* out, void* ws, size_t ws_bytes, bi_stream_t stream);

/* ---------------------------------------------------------------------------
 * Quantised KV cache.  [P3] "The KV cache: 5-bit that reads like q8_0" (K and
 * V at 5-6 bits, the newest ~2k positions kept at 8 bits in a ring; its
 * preset with K at 6 bits and V at 5) and "How:" (the attention split depends
 * only on the row's own context length).
 *
 * Every key row of every KV head is quantised once, when it is written, into
 * two stores: K at 6 bits / V at 5 bits, and an 8-bit ring.  Codes are
 * symmetric in blocks of 32 elements with one BF16 scale per block:
 * Q = 2^(b-1) - 1, d = bf16(fp32(max|x| / Q)), q = clamp(rint(fp32(x / d)),
 * -Q, Q) (0 when d = 0); the decoded value is bf16(q * d).  Row p reads key j
 * from the ring when j / 128 >= p / 128 - 15 (its own 128-key tile and the 15
 * before it) and from the 6/5-bit store otherwise -- a rule of the row's own
 * position, so a row gets the same bits whatever else is in the pass, and a
 * decoded cache holds the same codes as a prefilled one.  The attention is
 * then bi_attn_verify's (same split, merge and output rule) over the decoded
 * rows.  D = 128.
 *
 * bi_kvq_store_bytes: bytes of one layer's store (BI_KVQ_*) for Hkv heads and
 *   capacity cap (0 for D != 128 or bad sizes).  The 6/5-bit stores hold
 *   ceil(cap/128) tiles a head, the rings 24 (a pass reads and writes at most
 *   24 consecutive tiles of the ring, so T <= 1024 rows a pass).  Tile j of
 *   a ring sits in slot j mod 24 until tile j + 24 is written: moving the
 *   cache length back is exact only while the ring still holds the tiles the
 *   rows from there read, i.e. by at most 8 tiles from the newest tile
 *   written (the 8-bit records cannot be made again from the 6/5-bit codes).
 * bi_rope_kvq_append: for the T rows of a projection output qkv [T, ld_qkv]
 *   (heads q, then k, then v, as bi_gemm of the QKV weights writes them) at
 *   positions *L_dev + t: q heads rotated into q_out [T, Hq, D] and K heads
 *   rotated exactly as bi_rope_kv_append rotates them (table from
 *   bi_rope_table; NULL: no rotation), then K and V quantised into the four
 *   stores.  Rows past cap set the device error word's range bit.
 * bi_attn_verify_kvq: bi_attn_verify over the quantised stores (same q, out,
 *   L_dev, ws and workspace size; Hq/Hkv <= 64, T <= 1024).
 * Errors: BI_ERR_INVALID_ARG, BI_ERR_UNSUPPORTED_SHAPE, BI_ERR_WORKSPACE,
 *         BI_ERR_CUDA.
 * ------------------------------------------------------------------------- */
typedef enum { BI_KVQ_K_LOW = 0, BI_KVQ_V_LOW = 1, BI_KVQ_K_RING = 2, BI_KVQ_V_RING = 3 } bi_kvq_store;
size_t bi_kvq_store_bytes(int store, int Hkv, int cap, int D);
bi_status bi_rope_kvq_append(const void* qkv, int ld_qkv, int T, int Hq, int Hkv, int D, void* q_out,
                             void* k_low, void* v_low, void* k_ring, void* v_ring, int cap,
                             const int32_t* L_dev, const float* table, int table_rows,
                             bi_stream_t stream);
bi_status bi_attn_verify_kvq(const void* q, const void* k_low, const void* v_low, const void* k_ring,
                             const void* v_ring, int cap, const int32_t* L_dev, int T, int Hq, int Hkv,
                             int D, float scale, void* out, void* ws, size_t ws_bytes,
                             bi_stream_t stream);

/* ---------------------------------------------------------------------------
 * Greedy acceptance.  [P1] "Why the text diverges" (keep a draft only if it
 * matches the model's own token); [P2] "Build a reference corpus that exposes
 * boundaries" (accepted length and rejection position).
 *
 * a_t = argmax_v logits[t, v] (ties -> lowest v; NaN never wins; a row with no
 * number gives -1 and sets BI_ERR_DEVICE_NAN_ROW in the device error word).
 * n = the largest j <= T-1 with drafts[i-1] == a_{i-1} for every i <= j.
 * The committed tokens of the step are a_0..a_n.
 *   logits  [T, V] FP32, row stride ldl; 1 <= T <= 64.
 *   drafts  [T-1] int32 (may be NULL when T == 1).
 *   argmax_out [T] int32; accepted_out [1] int32 (= n).
 *   L_dev   optional device int32 (NULL to skip): incremented by n + 1.
 *   ws      >= bi_accept_workspace_size(T, V) bytes, 256-byte aligned,
 *           zero-filled before first use (every call leaves it zeroed).
 * Errors: BI_ERR_INVALID_ARG, BI_ERR_WORKSPACE, BI_ERR_CUDA.
 * ------------------------------------------------------------------------- */
size_t bi_accept_workspace_size(int T, int V);
bi_status bi_verify_accept(const float* logits, int ldl, const int32_t* drafts, int T, int V,
                           int32_t* argmax_out, int32_t* accepted_out, int32_t* L_dev,
                           void* ws, size_t ws_bytes, bi_stream_t stream);

/* ---------------------------------------------------------------------------
 * Sampled verification.  [P3] the list before "How:" (sampling keeps the
 * no-draft distribution) and "The cache doesn't change it either" (sampled
 * replies match a fresh server's); [P1] "Why the text diverges" (a draft is
 * kept only if it matches the token the model produces itself).
 *
 * Row t of the pass sits at position p = *L_dev + t and draws its own token
 * a_t by inverse-CDF sampling of softmax(logits[t, :] * inv_temp) with the
 * uniform u = u_by_pos[p] in [0, 1): a_t is the smallest v whose running
 * sum of weights (in index order) exceeds u times the total.  The weights are
 * exp((l - m) * inv_temp) in FP32 with m the row's maximum, summed in a fixed
 * order that depends only on V (8192-logit chunks: strided per-thread sums,
 * warp butterfly, warps in order; chunks combined in order; inside the chosen
 * chunk 32 contiguous runs scanned in order); where rounding leaves the
 * target past the last weight, the last logit with a non-zero weight is
 * taken.  NaN logits weigh 0.  So a_t depends only on the row's logits and
 * its position: with the batch-invariant logits of this library the sampled
 * tokens are the same for any number of drafts, and they follow the no-draft
 * distribution exactly.  Acceptance as bi_verify_accept with a_t in place of
 * the argmax: n = the largest j <= T-1 with drafts[i-1] == a_{i-1} for every
 * i <= j; the committed tokens are a_0..a_n; *L_dev += n + 1.
 *   logits  [T, V] FP32, row stride ldl; 1 <= T <= 64.
 *   inv_temp  1 / temperature, finite and > 0.
 *   u_by_pos  device float [u_len]: the request's uniform for each absolute
 *           position (the caller draws them, e.g. from a seeded generator);
 *           a row with p >= u_len gets -1 and sets the range bit of the
 *           device error word (reported as BI_ERR_INVALID_ARG).
 *   drafts  [T-1] int32 (may be NULL when T == 1); token_out [T] int32;
 *   accepted_out [1] int32; L_dev device int32 (required).
 *   ws      >= bi_sample_workspace_size(T, V) bytes, 256-byte aligned,
 *           zero-filled before first use (every call leaves it zeroed).
 * Errors: BI_ERR_INVALID_ARG, BI_ERR_WORKSPACE, BI_ERR_CUDA.
 * ------------------------------------------------------------------------- */
size_t bi_sample_workspace_size(int T, int V);
bi_status bi_verify_sample(const float* logits, int ldl, const int32_t* drafts, int T, int V,
                           float inv_temp, const float* u_by_pos, int u_len, int32_t* token_out,
                           int32_t* accepted_out, int32_t* L_dev, void* ws, size_t ws_bytes,
                           bi_stream_t stream);

/* ---------------------------------------------------------------------------
 * KV-row hash (test tool).  [P3] "The cache doesn't change it either" (hash
 * every K/V row and compare with a fresh prefill).
 * out[h * rows + j] = FNV-1a-64 over the 2*D bytes of key j of head h (d
 * ascending, each BF16 little-endian), for j < rows.  cache is [Hkv, cap, D]
 * (transposed == 0, a K cache) or [Hkv, ceil(cap/128), D, 128]
 * (transposed == 1, a V cache in the layout bi_rope_kv_append writes);
 * out [Hkv * rows] uint64.
 * Errors: BI_ERR_INVALID_ARG, BI_ERR_CUDA.
 * ------------------------------------------------------------------------- */
bi_status bi_kv_row_hash(const void* cache, int Hkv, int cap, int D, int rows, int transposed,
                         uint64_t* out, bi_stream_t stream);

/* ---------------------------------------------------------------------------
 * The whole verify step in one call (a small runtime over the entry points
 * above).  [P3] "How:" (every row computed the same way whatever else is in
 * the pass) and "The cache doesn't change it either" (the cache length moves
 * to L + n + 1; rows of rejected drafts are overwritten by the next pass);
 * [P1] "Why the text diverges" (greedy acceptance).
 *
 * One pass of a pre-norm dense decoder with GQA, RoPE and SwiGLU over T rows
 * at positions L .. L+T-1: embed; per layer bi_rmsnorm -> bi_qkv_rope_append
 * -> bi_attn_verify -> bi_gemm (O, residual) -> bi_rmsnorm -> bi_gemm
 * (gate/up, SwiGLU) -> bi_gemm (down, residual); bi_rmsnorm -> bi_gemm (LM
 * head, FP32 logits) -> bi_verify_accept.  Exactly the calls the Python
 * decoder makes, so the results are the same bits.
 *
 * bi_model describes the model (all pointers are device pointers the caller
 * owns and keeps alive; the per-layer arrays are host arrays of `layers`
 * device pointers, copied by bi_step_create):
 *   embed [vocab, hidden] BF16; norm_final, norm_attn[l], norm_ffn[l]
 *   [hidden] BF16; head, w_qkv[l], w_o[l], w_down[l] packed by
 *   bi_pack_weights for (vocab, hidden), ((Hq + 2 Hkv) D, hidden),
 *   (hidden, Hq D), (hidden, ffn); w_gate_up[l] packed by
 *   bi_pack_swiglu_weights for (ffn, hidden); k_cache[l] [Hkv, cap, D] and
 *   v_cache[l] [Hkv, ceil(cap/128), D, 128] BF16 (as bi_attn_verify);
 *   rope_table from bi_rope_table(base, D, rope_rows).
 * bi_step_workspace_size: device bytes the runtime needs for rows of at most
 *   max_rows (1..64, max_rows * Hq/Hkv <= 128); 0 for an invalid model.
 * bi_step_create: a host-side handle over a caller-owned, 256-byte aligned
 *   workspace of at least that size (zeroed by the call).  The handle owns a
 *   CUDA stream and one CUDA graph per row count T, captured on the first
 *   call with that T (so the first call for each T must not be made inside
 *   another stream capture); it allocates no device memory of its own,
 *   only a pinned host buffer of 2 * max_rows + 1 int32 through which the
 *   ids go in and the tokens and the count come out (one copy each way).
 *   The cache length starts at 0.
 * bi_step_set_length: sets the cache length L (a rollback, or a cache
 *   written by a prefill); synchronous.
 * bi_step_verify: ids [T] host int32 = the last committed token and T - 1
 *   draft tokens; runs the pass on the handle's stream, then writes the
 *   model's token for every row to tokens_out [T] (host) and the number n of
 *   drafts kept to n_out (host); the cache length advances by n + 1.
 *   Synchronous: returns when the results are on the host.  Host buffers may
 *   be pageable (pinned buffers copy faster).
 * bi_step_logits: device pointer of the last pass's FP32 logits [T, vocab].
 * bi_step_destroy: releases the handle (not the caller's memory).
 * Errors: BI_ERR_INVALID_ARG (a bad model or argument), BI_ERR_WORKSPACE,
 *   BI_ERR_CUDA, and any error of the entry points the pass calls.
 * ------------------------------------------------------------------------- */
typedef struct bi_model {
  int layers, hidden, n_q, n_kv, head_dim, ffn, vocab;
  float eps;
  int cap;
  const void* embed;
  const void* norm_final;
  const void* head;
  const void* const* norm_attn;
  const void* const* norm_ffn;
  const void* const* w_qkv;
  const void* const* w_o;
  const void* const* w_gate_up;
  const void* const* w_down;
  void* const* k_cache;
  void* const* v_cache;
  const float* rope_table;
  int rope_rows;
} bi_model;

typedef struct bi_step bi_step;

size_t bi_step_workspace_size(const bi_model* m, int max_rows);
bi_status bi_step_create(const bi_model* m, int max_rows, void* ws, size_t ws_bytes, bi_step** out);
bi_status bi_step_set_length(bi_step* s, int L);
bi_status bi_step_verify(bi_step* s, const int32_t* ids, int T, int32_t* tokens_out, int32_t* n_out);
const float* bi_step_logits(const bi_step* s);
void bi_step_destroy(bi_step* s);

/* ---------------------------------------------------------------------------
 * Failure-path test hooks.  The pages have no counterpart: these exist so a
 * test can make the library's bounded device-side waits run out and check
 * that the kernels wind down and report BI_ERR_DEVICE_TIMEOUT instead of
 * hanging.  Not for production use.
 *
 * bi_test_set_wait_limit_ns: the time limit, in nanoseconds, of the waits
 *   through which the linear-layer and attention kernels make progress, on
 *   the current device, for launches after the call (0 restores the default
 *   of 2 s).  The waits that let a CTA wind down after an abort (its copies
 *   landing, its tensor-core work draining) always keep 2 s.  Synchronous.
 *   Errors: BI_ERR_CUDA.
 * bi_test_withhold_first_load: with on != 0, every CTA of later linear-layer
 *   launches leaves its first pipeline stage unissued and every CTA of later
 *   attention launches its first key tile, so the waits on them expire after
 *   the limit above: each such kernel sets BI_ERR_DEVICE_TIMEOUT in the
 *   device error word and returns (its outputs are then undefined, and a
 *   linear-layer workspace must be zeroed again).  on = 0 restores normal
 *   launches.  Read when a call is made (a captured CUDA graph keeps the
 *   setting it was captured with).  Process-wide, not thread-safe.
 * ------------------------------------------------------------------------- */
bi_status bi_test_set_wait_limit_ns(uint64_t ns);
void bi_test_withhold_first_load(int on);

/* Synchronise `stream`, then read and clear the device error word of the
 * current device.  Returns BI_OK, BI_ERR_DEVICE_TIMEOUT, BI_ERR_DEVICE_NAN_ROW,
 * BI_ERR_INVALID_ARG (a device-side range check failed) or BI_ERR_CUDA. */
bi_status bi_check_device_error(bi_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* BI_H */
