/*
 * attn.h - C ABI of the GB300 (sm_103a) causal streaming-softmax attention
 * library, libattn.so.
 *
 * The method (StreamingAttentionSM86.alpha, lsalpha source view):
 *   forward   module header: for every 64-key block the running base-2 row
 *             maximum m, row sum l and fp32 weighted sum O are rescaled by
 *             2^(m - m') and the block's P V added; O / l is the output and
 *             L = m + log2 l the base-2 log-sum-exp.  Scores are taken in
 *             base 2 as t = S c, c = fp32-nearest(scale / ln 2); P is rounded
 *             to binary16 before its product with V; sums stay binary32.
 *   backward  header of the backward pass: P = 2^(S c - L), dP = dO V^T,
 *             D = rowsum(dO * O), dS = P (dP - D), dQ = s dS K,
 *             dK = s dS^T Q, dV = P^T dO (s = the natural scale), with no
 *             atomics (deterministic), split as the page-1 header of
 *             streamingAttentionRowTermsOrderedUncheckedSM86 describes: row
 *             terms, then a key pass that stores dS, then dQ from stored dS.
 *   lengths   gist self_attn_fwd (snippet.py): query rows and keys at or past
 *             a sequence's length are masked; such rows output zero.
 *
 * Layouts (the pages' planes with a leading batch index added), all dense
 * row-major, element sizes in brackets:
 *   q, dout   [B][H][T][64]      binary16 (uint16_t bit patterns)
 *   k         [B][Hkv][T][64]    binary16
 *   vt        [B][Hkv][64][T]    binary16 (V transposed)
 *   o         [B][T][H*64]       binary16 (token-major, heads merged)
 *   lse,delta [B][H][T]          binary32 (lse in base 2)
 *   dq        [B][H][T][64]      binary32
 *   dk        [B][Hkv][T][64]    binary32 (summed over each K/V head's group)
 *   dvt       [B][Hkv][64][T]    binary32 (dV transposed, unscaled)
 * Query head h reads K/V head h / (H / Hkv).
 *
 * Ownership: the caller allocates every buffer (device memory) and the
 * backward workspace; the library allocates no device memory (only tensor
 * memory inside its kernels) and keeps no state beyond cached per-device
 * properties.  Every call is asynchronous on the given stream (a
 * cudaStream_t passed as void*; NULL is the legacy default stream) and
 * returns after the launch.
 *
 * Errors: every entry point validates its arguments on the host before any
 * launch and returns one of the ATTN_ codes below; nothing is launched when
 * the result is not ATTN_OK.  Device-side failures (a bounded wait that ran
 * out) are reported by attn_last_device_error.
 */
#ifndef CSS_ATTN_H
#define CSS_ATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

enum {
  ATTN_OK = 0,
  ATTN_ERR_SHAPE = -1,          /* shape outside the admission rules below   */
  ATTN_ERR_NULL = -2,           /* a required pointer is NULL                */
  ATTN_ERR_ALIGN = -3,          /* a buffer is not 16-byte aligned           */
  ATTN_ERR_WORKSPACE = -4,      /* workspace smaller than required           */
  ATTN_ERR_CUDA = -5,           /* a CUDA runtime/driver call failed         */
  ATTN_ERR_DEVICE_TIMEOUT = -6, /* a kernel's bounded wait ran out           */
  ATTN_ERR_DEVICE = -7,         /* the current device is not sm_103          */
  ATTN_ERR_SCRATCH_LIMIT = -8   /* attn_bwd_noalloc: problem exceeds its
                                   static scratch                            */
};

/* Size of the static device scratch that attn_bwd_noalloc works in. */
#define ATTN_NOALLOC_SCRATCH_BYTES ((size_t)128 << 20)

/*
 * Problem shape.  Admission (the pages' admission predicate, "the program"
 * section of StreamingAttentionSM86.alpha): seq > 0 and a multiple of 64,
 * heads a multiple of kv_heads, heads <= 65535, head_dim == 64.  batch >= 1.
 * The pages' 32-bit byte-offset bound does not apply: offsets are 64-bit.
 *
 * seq_lens: NULL, or a DEVICE array [batch] of int32 lengths in 0..seq
 *   (values outside are clamped).  Query rows i >= len give O = 0,
 *   L = -inf, D = 0, dQ = 0; keys j >= len get dK = dV = 0.
 * causal: 1 masks keys after the query (the diagonal is kept); 0 attends to
 *   every key below the length.
 * scale: the natural score scale s; the kernels use c = fp32(s / ln 2).
 * head_begin, head_count: a chunk of K/V heads for attn_bwd_keys and
 *   attn_bwd_queries (with all their query heads); 0, 0 means all.  The
 *   workspace holds the chunk only, so a caller can bound it (or keep it
 *   L2-resident) by walking the heads in chunks.  attn_fwd and
 *   attn_row_terms ignore the chunk.
 * v_rows: 0: every `vt` argument is V^T, [B][Hkv][64][T] (the pages' forward
 *   layout); 1: it is V as rows, [B][Hkv][T][64] (K's layout, the pages'
 *   backward layout and their row-V forward), so no transposed copy of V
 *   is needed.  Results are the same either way.  Other values:
 *   ATTN_ERR_SHAPE.
 */
typedef struct attn_shape {
  int32_t batch;
  int32_t seq;
  int32_t heads;
  int32_t kv_heads;
  int32_t head_dim;
  int32_t causal;
  const int32_t* seq_lens;
  float scale;
  int32_t head_begin;
  int32_t head_count;
  int32_t v_rows;
} attn_shape;

/*
 * Forward pass (forward module header; "one key tile" and epilogue
 * sections).  Reads q, k, vt; writes o and lse.  All pointers device,
 * 16-byte aligned.
 */
ATTN_API int attn_fwd(const attn_shape* shape, const uint16_t* q, const uint16_t* k,
             const uint16_t* vt, uint16_t* o, float* lse, void* stream);

/*
 * Row terms D = rowsum(dO * O) (streamingAttentionRowTermsOrderedUncheckedSM86,
 * page 1): the stored binary16 O and dO widened, summed in binary32.
 * Reads o and dout; writes delta [B][H][T].  Device pointers, 16-byte aligned.
 */
ATTN_API int attn_row_terms(const attn_shape* shape, const uint16_t* o,
                   const uint16_t* dout, float* delta, void* stream);

/*
 * Bytes of the dS workspace that attn_bwd_keys writes and attn_bwd_queries
 * reads for this shape and head chunk (0 if the shape is invalid).  The
 * layout inside is private to the library: per (batch, query head of the
 * chunk, 128-query block, 128-key block) one 32 KiB binary16 tile of dS^T,
 * causal shapes storing only blocks on or below the diagonal.
 */
ATTN_API size_t attn_bwd_workspace_bytes(const attn_shape* shape);

/*
 * Key pass (key launch of StreamingAttentionSM86.alpha, with the score
 * gradients stored as the page-1 header describes).  For each 128-key block
 * of each K/V head in the chunk and each query block that can see it:
 * S^T = K Q^T, P^T = 2^(S^T c - L), dP^T = V dO^T, dS^T = P^T (dP^T - D);
 * dV += P^T dO and dK += dS^T Q over every query head of the group; dS^T is
 * stored (binary16) into ds_ws.  Writes dk = s * sum and dvt (unscaled) for
 * the chunk's K/V heads.  Needs lse from attn_fwd and delta from
 * attn_row_terms (or attn_bwd_queries_fused).  ds_ws: device, ws_bytes >=
 * attn_bwd_workspace_bytes; or ds_ws = NULL with ws_bytes = 0, in which case
 * dS is not stored (for callers that take dQ from attn_bwd_queries_fused).
 */
ATTN_API int attn_bwd_keys(const attn_shape* shape, const uint16_t* q, const uint16_t* k,
                  const uint16_t* vt, const uint16_t* dout, const float* lse,
                  const float* delta, void* ds_ws, size_t ws_bytes, float* dk,
                  float* dvt, void* stream);

/*
 * dQ pass (streamingAttentionQueryFromScores section): for each 128-query
 * block, dQ = s * sum over visible key blocks of dS K, dS read from the
 * workspace attn_bwd_keys filled for the same shape and chunk.  Writes dq
 * for the chunk's query heads.
 */
ATTN_API int attn_bwd_queries(const attn_shape* shape, const uint16_t* k,
                     const void* ds_ws, size_t ws_bytes, float* dq,
                     void* stream);

/*
 * Fused query pass (the query launch streamingAttentionQuerySM86 of
 * StreamingAttentionSM86.alpha, backward-pass header, which forms D for its
 * rows from dO and the forward's O, writes it for the key launch, and walks
 * the query tile's key tiles forming S, P and dP again): for each 128-query
 * block, D = rowsum(dO * O) (stored binary16 O widened, binary32 sum) is
 * written to delta, then S = Q K^T, P = 2^(S c - L), dP = dO V^T and
 * dS = P (dP - D) are recomputed for every visible key block and
 * dQ = s * sum of dS K is accumulated; dS is rounded to binary16 before its
 * product, as in the key pass.  Needs no workspace and replaces
 * attn_row_terms: call it after attn_fwd and before
 * attn_bwd_keys(..., NULL, 0, ...), which reads the delta it wrote.  It
 * recomputes two products per tile pair to avoid the dS workspace, whose
 * size and traffic grow as T^2 (2 B per visible (query, key) pair and head).
 * Reads q, k, vt, dout, o (token-major, from attn_fwd) and lse; writes delta
 * and dq for the chunk's query heads (rows past a sequence's length: D = 0,
 * dQ = 0).  Device pointers, 16-byte aligned, layouts as above.
 */
ATTN_API int attn_bwd_queries_fused(const attn_shape* shape, const uint16_t* q,
                                    const uint16_t* k, const uint16_t* vt,
                                    const uint16_t* dout, const uint16_t* o, const float* lse,
                                    float* delta, float* dq, void* stream);

/*
 * Device buffers of one whole problem, as attn_step_host uses them.  All
 * device pointers, 16-byte aligned, laid out as the calls above state:
 * q, dout [B][H][T][64] and k [B][Hkv][T][64], vt [B][Hkv][64][T] (binary16);
 * o [B][T][H*64] (binary16); lse, delta [B][H][T]; dq [B][H][T][64],
 * dk [B][Hkv][T][64], dvt [B][Hkv][64][T] (binary32); ws the dS workspace of
 * ws_bytes >= attn_bwd_workspace_bytes, or NULL with 0 bytes (attn_step_host
 * then uses the fused query pass).  Owned by the caller.
 */
typedef struct attn_device_buffers {
  uint16_t* q;
  uint16_t* k;
  uint16_t* vt;
  uint16_t* dout;
  uint16_t* o;
  float* lse;
  float* delta;
  void* ws;
  size_t ws_bytes;
  float* dq;
  float* dk;
  float* dvt;
} attn_device_buffers;

/*
 * attn_step_host - one whole forward and backward from host memory to host
 * memory: copies h_q, h_k, h_vt, h_dout into the device buffers, runs
 * attn_fwd, attn_row_terms, attn_bwd_keys and attn_bwd_queries, and copies
 * O, L, dQ, dK and dV^T back into h_o, h_lse, h_dq, h_dk, h_dvt (layouts as
 * in attn_device_buffers).  The method's pages have no host-transfer step;
 * this is the library's runtime around the path.  The copies overlap the
 * kernels: dO goes in while the forward runs, O and L come out during the
 * backward, dK and dV^T during the dQ pass, and dQ in two halves, the first
 * while the second is computed; a second stream owned by the library (one
 * per device) carries them, and `stream` waits for it before the call's work
 * ends.  Asynchronous: returns once everything is enqueued; the host outputs
 * are valid after `stream` completes, and no host buffer may be touched
 * before then.  Host buffers should be page-locked (pageable memory works,
 * but its copies do not overlap).  The shape must cover every K/V head
 * (head_begin = 0, head_count = 0 or Hkv); seq_lens, if any, is a device
 * array.  The step takes dQ from attn_bwd_queries_fused, run before a key
 * pass that stores no dS (no workspace needed), when dev->ws = NULL and
 * dev->ws_bytes = 0, and also when dQ (B*H*T*64*4 bytes) is 8 MiB or more:
 * dQ is then ready before the key pass and its copy back overlaps it, which
 * measured faster end to end on every such workload (the host link bounds
 * the step); smaller problems use the workspace and the stored order.
 * Errors as the calls above; a CUDA failure while enqueueing
 * returns ATTN_ERR_CUDA with the work enqueued so far left on the streams.
 */
ATTN_API int attn_step_host(const attn_shape* shape, const attn_device_buffers* dev,
                            const uint16_t* h_q, const uint16_t* h_k, const uint16_t* h_vt,
                            const uint16_t* h_dout, uint16_t* h_o, float* h_lse, float* h_dq,
                            float* h_dk, float* h_dvt, void* stream);

/*
 * attn_step_host_order - which order attn_step_host takes for this shape and
 * these buffers: ATTN_STEP_STORED (row terms, the key pass storing dS, the dQ
 * pass) or ATTN_STEP_FUSED (the fused query pass, then the key pass storing
 * no dS).  Host only (nothing is launched or dereferenced but the two
 * structs); ATTN_ERR_SHAPE or ATTN_ERR_NULL as attn_step_host would return.
 */
enum { ATTN_STEP_STORED = 0, ATTN_STEP_FUSED = 1 };
ATTN_API int attn_step_host_order(const attn_shape* shape, const attn_device_buffers* dev);

/*
 * dQ pass with the inverse half-split rotation in its epilogue (the rotated
 * form of the dQ-from-scores pass in StreamingAttentionSM86.alpha, the
 * epilogue that turns dQ back by the inverse rotation and stores the QKV
 * pullback's bfloat16 operand): as attn_bwd_queries, but each query row
 * p of head h, x = s * sum, is written as
 *   out[c]      = x[c] cos[p][c] + x[c + 32] sin[p][c]
 *   out[c + 32] = x[c + 32] cos[p][c] - x[c] sin[p][c]      (c < 32)
 * (each sine product rounded to binary32 before the fused multiply-add),
 * rounded to bfloat16, at dq_out[(b T + p) ld + 64 h + c]: token-major, so
 * the output can be a column block of a wider [B][T][width] projection
 * gradient (pass its first column and ld = width).  cos_tab, sin_tab:
 * device [T][32] binary32.  ld >= heads * 64 and a multiple of 8
 * (ATTN_ERR_SHAPE otherwise); device pointers, 16-byte aligned.  The
 * chunk's query heads are written; rows past a sequence's length get 0.
 */
ATTN_API int attn_bwd_queries_rotated(const attn_shape* shape, const uint16_t* k,
                                      const void* ds_ws, size_t ws_bytes, const float* cos_tab,
                                      const float* sin_tab, uint16_t* dq_out, int64_t ld,
                                      void* stream);

/*
 * A token-major block of a fused projection's gradient: the gradient row of
 * sequence position t and head `head` (64 columns) lives at
 * [(b T + t) ld + 64 head + c] of f32 (binary32) and of bf16 (bfloat16,
 * rounded to nearest even from the binary32 value); a NULL pointer is not
 * written, one of the two must be given.  Point the pointers at the block's
 * first column inside the wider [B][T][width] gradient and pass ld = width.
 * ld >= heads * 64 and a multiple of 8 (ATTN_ERR_SHAPE otherwise); both
 * pointers 16-byte aligned (ATTN_ERR_ALIGN).
 */
typedef struct attn_projection {
  float* f32;
  uint16_t* bf16;
  int64_t ld;
} attn_projection;

/*
 * Key pass with the projection-fused epilogue (StreamingAttentionSM86.alpha,
 * the key launch's epilogue that stores dK = s * sum and dV straight into a
 * fused projection's gradient, token-major, binary32 and bfloat16, instead
 * of the [head][T][64] dK and [head][64][T] dV^T planes a layout pass then
 * converted): as attn_bwd_keys, but dK goes to dk_out and dV (row = key
 * position, not transposed) to dv_out, each with one 64-column block per
 * K/V head.  ds_ws may be NULL with ws_bytes 0 (no dS store), as there.
 */
ATTN_API int attn_bwd_keys_projected(const attn_shape* shape, const uint16_t* q,
                                     const uint16_t* k, const uint16_t* vt,
                                     const uint16_t* dout, const float* lse,
                                     const float* delta, void* ds_ws, size_t ws_bytes,
                                     const attn_projection* dk_out,
                                     const attn_projection* dv_out, void* stream);

/*
 * dQ pass with the projection-fused epilogue (StreamingAttentionSM86.alpha,
 * the dQ epilogue that stores dQ = s * sum straight into a fused
 * projection's gradient, token-major, binary32 and bfloat16): as
 * attn_bwd_queries, but dQ goes to dq_out, one 64-column block per query
 * head.
 */
ATTN_API int attn_bwd_queries_projected(const attn_shape* shape, const uint16_t* k,
                                        const void* ds_ws, size_t ws_bytes,
                                        const attn_projection* dq_out, void* stream);

/*
 * attn_bwd_noalloc - the key pass and the dQ pass (what attn_bwd_keys and
 * then attn_bwd_queries compute) without a caller-supplied workspace.  The
 * method's pages have no counterpart to this entry point.  It is for callers
 * that may not allocate device memory while they run: for example a plugin
 * or custom-operator interface whose execute step must not allocate because
 * the host framework owns all device memory, or a latency-bound loop that
 * cannot take the implicit device synchronisation of cudaMalloc.
 *
 * The dS scratch lives in a static device array of
 * ATTN_NOALLOC_SCRATCH_BYTES (128 MiB) inside the library; every GPU on
 * which the library's code is loaded holds that array until the process
 * exits.  The call walks the chunk's K/V heads in groups that fit the array,
 * and calls no cudaMalloc, cudaFree or other allocating routine.  The first
 * call in a device's context looks up the array's device address (with that
 * device current) and keeps it for that context; after a device reset the
 * next call looks it up again.  Make the first call on each device before
 * any stream capture.
 *
 * Arguments as attn_bwd_keys and attn_bwd_queries (device pointers, 16-byte
 * aligned, layouts in the file header): reads q, k, vt, dout, lse, delta;
 * writes dq, dk, dvt for the K/V heads of the shape's head chunk (0, 0 = all)
 * and their query heads.  Returns ATTN_ERR_SCRATCH_LIMIT, before launching
 * anything, when one K/V head's share (batch x query heads per K/V head x
 * dS tiles of one head x 32 KiB) exceeds the array; other errors as the
 * other entry points.
 *
 * Every call, on every stream and host thread, shares the one array, and a
 * call leaves its dS tiles there.  Nothing in the array has to start at
 * zero: each tile the dQ pass reads was written earlier in the same call.
 * Calls whose work overlaps on the GPU race on the array and give wrong
 * results: order them on one stream or synchronise between them.
 */
ATTN_API int attn_bwd_noalloc(const attn_shape* shape, const uint16_t* q,
                              const uint16_t* k, const uint16_t* vt,
                              const uint16_t* dout, const float* lse,
                              const float* delta, float* dq, float* dk,
                              float* dvt, void* stream);

/* A static, human-readable message for an ATTN_ code. */
ATTN_API const char* attn_error_string(int code);

/*
 * Synchronises the stream, then reports and clears the current device's
 * device-side error word: ATTN_OK, or ATTN_ERR_DEVICE_TIMEOUT when a kernel
 * gave up a bounded wait (its outputs are then undefined).  ATTN_ERR_CUDA if
 * the synchronisation itself failed.
 */
ATTN_API int attn_last_device_error(void* stream);

/*
 * Sets the time limit of every bounded wait inside the kernels launched
 * afterwards on any device (nanoseconds; 0 restores the default of 2 s).
 * Values below ATTN_MIN_WAIT_LIMIT_NS (10 ms) are raised to it, so that no
 * ordinary pipeline wait gives up on a busy GPU.  The waits that drain a
 * kernel's own copies and products before it frees tensor memory or exits
 * keep their own fixed limit, whatever is set here.  Not part of the method:
 * a safety bound so that a kernel never spins forever.
 */
#define ATTN_MIN_WAIT_LIMIT_NS ((uint64_t)10000000)
ATTN_API void attn_set_wait_limit_ns(uint64_t limit_ns);

/* The bounded-wait limit that kernels launched now would use (nanoseconds). */
ATTN_API uint64_t attn_wait_limit_ns(void);

/*
 * Self-test of the bounded wait: launches one block that waits on a barrier
 * nothing will complete, with a limit of limit_ns (its own, not the one set
 * above; 0 means 1 ms), then synchronises and returns what
 * attn_last_device_error reports (ATTN_ERR_DEVICE_TIMEOUT when the wait gave
 * up as it should).  The probe issues no copy or product, so its short limit
 * is safe.  Not part of the method.
 */
ATTN_API int attn_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/*
 * The CUDA runtime's message for the last CUDA call of this library that
 * failed on the calling host thread (the cause behind an ATTN_ERR_CUDA), or
 * "no error".  Diagnostic only.
 */
ATTN_API const char* attn_last_cuda_error(void);

/*
 * Self-test of the two arithmetic steps every kernel relies on (the
 * precision contract of the forward module header: P rounded to binary16
 * before its product with V, and P = 2^t): for device arrays x[n] (n even),
 * writes packed[i] = the binary16x2 word of (x[2i] low, x[2i+1] high),
 * rounded to nearest even, and e2[i] = 2^x[i] as the kernels compute it.
 * Synchronises the stream.  Not part of the method; for tests.
 */
ATTN_API int attn_selftest_arith(const float* x, uint32_t* packed, float* e2, int n,
                                 void* stream);

/* Library version, major * 10000 + minor * 100 + patch. */
ATTN_API int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CSS_ATTN_H */
