/*
 * libskipsm — Skip Softmax block-sparse attention for NVIDIA B300 (sm_103a).
 *
 * The operation ("Accelerating Long-Context Inference with Skip Softmax in
 * NVIDIA TensorRT-LLM", sections "Skip Softmax Mechanism" and "Detailed
 * Analysis"; "NVIDIA Introduces Skip Softmax for Enhanced LLM Inference
 * Efficiency", section "Understanding Skip Softmax"): FlashAttention-style
 * attention over key tiles with an online softmax.  For each (query tile,
 * key tile) visited in ascending key order, let m~_r be the tile's maximum of
 * the scaled logits in row r and m_r the running maximum of row r over the
 * tiles before it.  The tile is skipped — no exponentials, no P.V product —
 * when lambda > 0 and exp(m~_r - m_r) < lambda for every valid row r.  A
 * skipped tile cannot raise the running maximum (lambda <= 1), so the maximum
 * stays the exact prefix maximum.  lambda = 0 is exact dense attention.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are bf16, contiguous, D innermost:
 *      prefill  q, o : [B][Hq][Sq][D]     decode  q, o : [B][Hq][D]
 *               k, v : [B][Hkv][Skv][D]           k, v : [B][Hkv][Skv][D]
 *    Query head h reads kv head h / (Hq / Hkv).
 *  - All pointers are device pointers owned by the caller, 16-byte aligned.
 *    The library never frees them and allocates no device memory per call
 *    (tensor maps live in kernel parameters; the decode workspace is the
 *    caller's).
 *  - Calls only enqueue work on `stream` (a cudaStream_t, NULL = legacy
 *    default stream) and return.  Argument errors are detected on the host
 *    before any launch and return SKIPSM_ERR_INVALID_ARG / _UNSUPPORTED with
 *    nothing enqueued; skipsm_last_error() gives the reason (thread-local).
 *  - Device-side failures (a pipeline wait that exceeded its bound) set a
 *    device status word instead of trapping.  By default that is the library's
 *    one word per device (per CUDA context), shared by every stream and host
 *    thread: skipsm_check() reads and clears it for all of them, so with calls
 *    from several streams or threads a failure may be reported to, and cleared
 *    by, a caller other than the one whose launch timed out.  Such callers pass
 *    their own word in the `status` option of the _ex calls instead.
 *  - Softmax scale is 1/sqrt(D) unless an _ex call gives one.  Causal masking
 *    is bottom-right aligned: query i sits at key position Skv - Sq + i.
 *  - lambda must be finite and in [0, 1].
 *  - skip_counts, when not NULL, is a device array of Hq uint64 that the call
 *    zeroes (on `stream`) and fills: prefill — skipped (query tile, key tile)
 *    pairs per query head, summed over batch and query tiles; decode — skipped
 *    key tiles of each GQA group, summed over batch, repeated for each of the
 *    group's query heads (the decode vote is over the group's G heads).
 */
#ifndef SKIPSM_H
#define SKIPSM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SKIPSM_VERSION 108

typedef enum skipsm_status {
  SKIPSM_OK = 0,
  SKIPSM_ERR_INVALID_ARG = 1,  /* bad pointer, shape, lambda or option */
  SKIPSM_ERR_UNSUPPORTED = 2,  /* valid but not implemented (D, G, tiles) */
  SKIPSM_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
  SKIPSM_ERR_TIMEOUT = 4,      /* a kernel gave up on a bounded wait */
  SKIPSM_ERR_WORKSPACE = 5     /* decode workspace missing or too small */
} skipsm_status;

/* Library version (SKIPSM_VERSION of the build). */
int skipsm_version(void);

/* Message of the last failed call on this host thread ("" if none). */
const char* skipsm_last_error(void);

/*
 * Waits for `stream`, then reads and clears the library's device status word
 * (the one shared by every call on the current device that passed no `status`
 * option; see the conventions above).
 * *device_status (if not NULL) receives the raw word: 0 = clean, otherwise a
 * code identifying the wait that timed out.  Returns SKIPSM_ERR_TIMEOUT when
 * the word was set, SKIPSM_ERR_CUDA when synchronisation failed.
 */
skipsm_status skipsm_check(void* stream, int* device_status);

/* ------------------------------------------------------------------------ */
/* Prefill                                                                    */
/* ------------------------------------------------------------------------ */

/* Optional controls and outputs of a prefill call; zero-initialise. */
typedef struct skipsm_prefill_opts {
  int tile_q;             /* rows of one skip vote: 64 or 128; 0 = 64 if D == 64 else 128 */
  int tile_k;             /* keys per key tile: 64 or 128; 0 = 64 if D == 64 else 128 */
  float softmax_scale;    /* 0 = 1/sqrt(D) */
  float* lse;             /* optional out [B][Hq][Sq] fp32, natural-log LSE of the kept keys */
  uint8_t* skip_mask;     /* optional out [B][Hq][ceil(Sq/tile_q)][ceil(Skv/tile_k)]:
                             0 kept, 1 skipped, 2 not visited (causal) — fully written */
  uint64_t* visited_counts; /* optional out [Hq]: visited tile pairs per head (zeroed, filled) */
  int wait_limit_ms;      /* bound of each pipeline wait in the kernel; 0 = 2000 ms */
  int exp_mode;           /* weights of the kept tiles' keys:
                             0 = exact exponentials exp(s - m');
                             1 = Rowmax-PoT ("Approximating Softmax in Pretrained LLMs: Model
                                 Sensitivity and Kernel Acceleration", AI Summary, Abstract):
                                 2^round((s - m') * log2 e), anchored at the running row max m'
                                 after the key's tile, 0 below 2^-126.5 (the skip vote is
                                 unchanged: it always uses the exact maxima);
                             other values: SKIPSM_ERR_INVALID_ARG */
  int qk_format;          /* element type of q and k: 0 = bf16; 1 = e4m3 (OCP FP8, 1 byte,
                             same [B][H][S][D] layouts, D = 128 and tile_k = 128 only) for the
                             FP8/BF16 mixed-precision path ("Approximating Softmax in Pretrained
                             LLMs: ...", AI Summary): Q.K^T runs as an e4m3 tcgen05 MMA with
                             fp32 accumulation, v, P and o stay bf16 */
  float qk_descale;       /* multiplies Q.K^T before the softmax scale (the product of the q and
                             k quantisation scales); 0 = 1 */
  const uint8_t* block_mask; /* optional in, device [B][Hq][ceil(Sq/tile_q)][ceil(Skv/tile_k)]:
                             nonzero = visit the (vote tile, key tile) pair.  Skip Softmax
                             combined with a prefill block selector ("NVIDIA Introduces Skip
                             Softmax ...", "Benefits and Implementation"): an unselected pair
                             takes no exponentials, no P.V, no vote and does not enter the
                             running max (its Q.K^T is still computed when the other vote
                             group or Q tile of the CTA needs the key tile); skip_mask reports
                             it as 2; a row with no visible selected key gets o = 0 and
                             lse = -inf.  NULL = every pair. */
  int inject_wait_timeout; /* failure-detection test hook: in every CTA the softmax warps first
                              wait on a barrier nothing arrives at (half of wait_limit_ms); the
                              kernel ends early, outputs are undefined and skipsm_check()
                              reports site 25 */
  int* status;            /* optional device int, 4-byte aligned, owned by the caller: this
                             call's kernels record a timed-out wait here (the site code, first
                             writer wins) instead of in the library's shared word.  The call
                             neither clears nor reads it: zero it before the call, read it after
                             the stream has finished.  NULL = the shared word (skipsm_check) */
  int v_format;           /* element type and layout of v: 0 = bf16 [B][Hkv][Skv][D];
                             1 = e4m3, transposed: [B][Hkv][D][Skv], keys innermost (the
                             K-major operand of the e4m3 tensor-core product; Skv a multiple
                             of 16), with qk_format = 1, D = 128, tile_k = 128 and
                             exp_mode = 0 only.  Then P.V runs in e4m3 too: on a kept tile each
                             weight p = exp(s - m') (m' the exact running row max after the
                             tile) enters it as e4m3(2^8 p) / 2^8, rounded to nearest even,
                             while the row sum keeps the fp32 p ("Approximating Softmax in
                             Pretrained LLMs: ...", AI Summary: FP8/BF16 mixed precision) */
  float v_descale;        /* with v_format = 1: multiplies the output (the caller's v
                             quantisation scale); 0 = 1 */
  int v_load;             /* when the kernel fetches a key tile's V rows ("NVIDIA Introduces Skip
                             Softmax ...", "Benefits and Implementation": a skipped block need
                             not be read): 0 = the library's choice (currently 1); 1 = every V
                             tile, ahead of the vote; 2 = only once a query tile of the CTA keeps
                             the key tile (bf16 v, D = 128, tile_k = 128, exp_mode = 0; other
                             configurations fall back to 1).  Results are identical. */
  int sync_check;         /* nonzero: the call waits for `stream` before it returns and reports
                             its kernels' device status — SKIPSM_ERR_TIMEOUT if a wait timed out
                             (the site is in skipsm_last_error()).  With `status` given it reads
                             that word and leaves it as it is; otherwise it reads and clears the
                             shared word, as skipsm_check() does.  0 = return once enqueued. */
} skipsm_prefill_opts;

/*
 * Skip Softmax prefill (self-attention over a prompt).
 *   q, k, v, o       device bf16 tensors, layouts above; o is written.
 *   B, Hq, Hkv       batch, query heads, kv heads (Hq % Hkv == 0)
 *   Sq, Skv          query / key lengths (>= 1; Sq <= Skv when causal)
 *   D                head dim: 64 or 128
 *   causal           nonzero = causal mask
 *   lambda           skip threshold in [0, 1]
 *   skip_counts      optional device uint64[Hq] (see above)
 * Returns SKIPSM_OK once the work is enqueued.
 */
skipsm_status skipsm_prefill(const void* q, const void* k, const void* v, void* o,
                             int B, int Hq, int Hkv, int Sq, int Skv, int D,
                             int causal, float lambda, uint64_t* skip_counts,
                             void* stream);

/* skipsm_prefill with tile overrides and optional outputs (opts may be NULL). */
skipsm_status skipsm_prefill_ex(const void* q, const void* k, const void* v, void* o,
                                int B, int Hq, int Hkv, int Sq, int Skv, int D,
                                int causal, float lambda, uint64_t* skip_counts,
                                const skipsm_prefill_opts* opts, void* stream);

/* ------------------------------------------------------------------------ */
/* Decode (one query token per sequence, split-KV + log-sum-exp combine)      */
/* ------------------------------------------------------------------------ */

/*
 * Number of KV splits a decode call uses when the caller asks for 0.  The
 * (b, kv head, split) CTAs run in waves of 2 per SM (the current device's SM
 * count; 148, the B300's, when no device can be queried); the default
 * is the count with the least modelled time, waves x (tiles per split + a
 * start-up of 4 tiles), taking the fewest splits on a tie and at least 16 key
 * tiles of 64 per split (every split keeps its first tile and restarts its
 * running max, so short splits cap the skip ratio).  The key range is cut into
 * ceil(nblk/splits)-tile splits, and empty trailing splits are dropped, so the
 * count returned here is the effective one.  Returns 0 for invalid sizes.
 */
int skipsm_decode_num_splits(int B, int Hkv, int Skv, int requested);

/*
 * Bytes of device workspace a decode call needs: per (b, query head, split)
 * a D-float partial output and one float log-sum-exp, 256-byte aligned.
 * num_splits = 0 selects the default.  Returns 0 for invalid sizes.
 */
size_t skipsm_decode_workspace_size(int B, int Hq, int Hkv, int Skv, int D, int num_splits);

/* Optional controls and outputs of a decode call; zero-initialise. */
typedef struct skipsm_decode_opts {
  int num_splits;         /* 0 = skipsm_decode_num_splits(B, Hkv, Skv, 0) */
  float softmax_scale;    /* 0 = 1/sqrt(D) */
  float* lse;             /* optional out [B][Hq] fp32 natural-log LSE */
  uint8_t* skip_mask;     /* optional out [B][Hkv][ceil(Skv/64)]: 0 kept, 1 skipped
                             (2 not selected, with block_mask) */
  int wait_limit_ms;      /* bound of each pipeline wait; 0 = 2000 ms */
  int inject_wait_timeout; /* failure-detection test hook: one split-kernel wait is made to
                              run out (nothing arrives on its barrier); the kernels end early,
                              outputs are undefined and skipsm_check() reports site 7 */
  const uint8_t* block_mask; /* optional in, device [B][Hkv][ceil(Skv/64)]: nonzero = visit
                              the 64-key tile.  Skip Softmax combined with a block selector
                              ("NVIDIA Introduces Skip Softmax ...", "Benefits and
                              Implementation"): tiles outside the mask are neither read nor
                              voted on and do not enter the running max; the skip rule runs over
                              the selected tiles of each split in ascending order; skip_mask
                              reports them as 2; a group with no selected tile gets o = 0 and
                              lse = -inf.  NULL = every tile.  With a mask each split's tile
                              list is kept in shared memory (2 bytes per tile of the split);
                              SKIPSM_ERR_UNSUPPORTED if it does not fit. */
  int* status;            /* optional per-call device status word, as in skipsm_prefill_opts */
  int sync_check;         /* nonzero: wait for `stream` and report the device status before
                             returning, as in skipsm_prefill_opts */
} skipsm_decode_opts;

/*
 * Skip Softmax decode step with GQA.  Key tiles are 64 keys; the skip vote of
 * a tile is over the G = Hq/Hkv query heads sharing the kv head, and a skipped
 * tile's V rows are never read from memory.
 *   q, o             device bf16 [B][Hq][D]
 *   k, v             device bf16 [B][Hkv][Skv][D] (the first Skv positions are valid)
 *   Hq/Hkv           G in {1, 2, 4, 8}
 *   D                64 or 128
 *   workspace        device buffer of >= skipsm_decode_workspace_size(...) bytes,
 *                    256-byte aligned, owned by the caller, not read before written
 * Launches a split kernel and a combine kernel on `stream`.
 */
skipsm_status skipsm_decode(const void* q, const void* k, const void* v, void* o,
                            int B, int Hq, int Hkv, int Skv, int D, float lambda,
                            uint64_t* skip_counts, void* workspace, size_t workspace_bytes,
                            void* stream);

/* skipsm_decode with split override and optional outputs (opts may be NULL). */
skipsm_status skipsm_decode_ex(const void* q, const void* k, const void* v, void* o,
                               int B, int Hq, int Hkv, int Skv, int D, float lambda,
                               uint64_t* skip_counts, void* workspace, size_t workspace_bytes,
                               const skipsm_decode_opts* opts, void* stream);

/* ------------------------------------------------------------------------ */
/* Threshold calibration                                                      */
/* ------------------------------------------------------------------------ */

/*
 * Picking lambda for a target skip ratio ("Accelerating Long-Context Inference
 * with Skip Softmax in NVIDIA TensorRT-LLM", "Impact on Accuracy vs. Speed": the
 * threshold trades speed against accuracy; "NVIDIA Introduces Skip Softmax ...",
 * "Accuracy and Sparsity Trade-offs": up to about 50% sparsity is near-lossless).
 *
 * The calibration runs the kernel at lambda values chosen by bisection on
 * log10(lambda) in [1e-9, 1] and returns the evaluated lambda whose measured
 * skip ratio is closest to `target_skip_ratio`.  The skip ratio cannot decrease
 * when lambda grows (a tile skipped at lambda is skipped at every larger lambda),
 * which is what makes bisection valid.  Each step synchronises `stream` to read
 * the counts.  The outputs of the last evaluated call are left in the buffers.
 */
typedef struct skipsm_calibration {
  float lambda;        /* chosen threshold */
  float skip_ratio;    /* skipped / visited tiles measured at that threshold */
  int launches;        /* attention calls made */
} skipsm_calibration;

/*
 * Prefill calibration.  Arguments as skipsm_prefill_ex; `counts` is caller-owned
 * device scratch of 2*Hq uint64 (skip counts, then visited counts).  target in
 * [0, 1]; max_iters in [1, 64] bisection steps (0 = 14).  opts->skip_mask,
 * opts->visited_counts and opts->lse must be NULL (opts may be NULL).
 */
skipsm_status skipsm_prefill_calibrate(const void* q, const void* k, const void* v, void* o,
                                       int B, int Hq, int Hkv, int Sq, int Skv, int D,
                                       int causal, float target_skip_ratio, int max_iters,
                                       uint64_t* counts, const skipsm_prefill_opts* opts,
                                       skipsm_calibration* result, void* stream);

/*
 * Decode calibration.  Arguments as skipsm_decode_ex; the skip ratio is skipped
 * 64-key tiles over all (b, kv head) tiles.  `counts` is device scratch of Hq
 * uint64.  opts->skip_mask and opts->lse must be NULL (opts may be NULL).
 */
skipsm_status skipsm_decode_calibrate(const void* q, const void* k, const void* v, void* o,
                                      int B, int Hq, int Hkv, int Skv, int D,
                                      float target_skip_ratio, int max_iters, uint64_t* counts,
                                      void* workspace, size_t workspace_bytes,
                                      const skipsm_decode_opts* opts,
                                      skipsm_calibration* result, void* stream);

/* ------------------------------------------------------------------------ */
/* Decode without a caller-provided workspace                                 */
/* ------------------------------------------------------------------------ */

/* Bytes of device memory the library keeps for skipsm_decode_noalloc. */
#define SKIPSM_DECODE_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * skipsm_decode for callers that cannot allocate device memory — for example a
 * plugin running inside a host framework that owns every device allocation, or
 * a serving loop that must never call cudaMalloc (it can synchronise the device).
 * The Skip Softmax pages have no counterpart of this call: it changes only where
 * the split-KV partial results are kept.
 *
 * Arguments, layouts, results and errors are those of skipsm_decode with the
 * default number of splits, minus the workspace.  The partials live in one
 * SKIPSM_DECODE_NOALLOC_SCRATCH_BYTES (16 MiB) array of device memory owned by
 * the library; every GPU that loads the library holds it until the process
 * exits.  A shape whose workspace, skipsm_decode_workspace_size(B, Hq, Hkv,
 * Skv, D, 0), is larger than that is rejected with SKIPSM_ERR_WORKSPACE
 * (skipsm_last_error() names the bytes needed) and nothing is launched.
 * Nothing is allocated or freed by the call.
 *
 * All calls share the array and it keeps what the last call left in it; no
 * part of it needs to start at zero.  Calls that can overlap on the GPU (other
 * streams, other host threads) race on it: the caller must order them.  The
 * first call on a device looks up the array's device address with that device
 * current; make that first call before any stream capture on the device.
 */
skipsm_status skipsm_decode_noalloc(const void* q, const void* k, const void* v, void* o,
                                    int B, int Hq, int Hkv, int Skv, int D, float lambda,
                                    uint64_t* skip_counts, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SKIPSM_H */
