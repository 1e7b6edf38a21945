/*
 * mla_gb300.h -- C ABI of the GB300 (sm_103a) MLA paged-decode library.
 *
 * Operation.  Multi-head latent attention decode in absorbed form over a
 * page-size-1 latent KV cache, for a block of T query tokens per request:
 *   - every KV entry is one 576-wide latent row (512 latent + 64 RoPE) shared
 *     by all heads; scores use all 576 columns, the output lives in the first
 *     512 ("[ROCm] Dspark MLA module", Details: absorb BMM, MLAAttention,
 *     concat_and_cache_mla);
 *   - each request's entries are a flat index list kv_indices[kv_indptr[b] ..
 *     kv_indptr[b+1]) into the pool ("[ROCm][Spec Decode] Add Aiter MLA decode
 *     support non-causal draft block", Purpose);
 *   - the block is either non-causal (every token sees all committed entries,
 *     same page, Purpose) or causal on global positions, including a
 *     round-robin context-parallel shard whose global lengths come from
 *     g_kv_indptr, and the call returns the log-sum-exp ("Speculative decode +
 *     DCP on gfx1250", Problem);
 *   - the pool is bf16 or fp8 e4m3fn with one per-tensor scale ("[ROCm][Spec
 *     Decode] ...", section "Three pieces");
 *   - long rows are split over the KV and merged through the LSE inside the
 *     call, driven by a split plan that is deterministic in its inputs so a
 *     CUDA-graph replay agrees with its capture; the plan is built on the host
 *     once from capacities (STATIC) or from the real lengths (HOST), or rebuilt
 *     on the device from the real lengths at every call (DYNAMIC) ("[DSV4] Tuned
 *     ASM FP8 decode with split plans; HCA on aiter's persistent V4-NM kernel",
 *     Summary parts 1 and 2);
 *   - an entry may carry its own global position and causal rows may have a
 *     sliding window, for the index lists of that page's layer types.
 *
 * The steps either side of the decode have their own entry points, declared
 * at the end: mla_cache_write and mla_rope_q_cache (new tokens into the cache,
 * q assembled for the decode) and mla_absorb_bmm (the per-head products that
 * take q into, and O out of, the latent space).
 *
 * Definition, for request b, token t in [0,T_b), head h:
 *   k_i = dec(pool[kv_indices[kv_indptr[b]+i]]) * kappa   (kappa = kv_scale for fp8, else 1)
 *   s_i = softmax_scale * <q[t,h,0:576], k_i[0:576]>
 *   visible(i) = !causal || base_b + i*pos_stride <= Lg_b - T_b + t
 *   LSE[t,h] = ln sum_{visible} exp(s_i)      O[t,h,:] = sum exp(s_i - LSE) k_i[0:512]
 *   no visible entry: O = 0, LSE = -inf.
 * base_b = pos_base_per_req[b] if given, else pos_base; Lg_b = g_kv_indptr[b+1] -
 * g_kv_indptr[b] if given, else the local length L_b.
 *
 * Layouts (row-major, contiguous):
 *   q        bf16 [total_q, H, 576]        total_q = qo_indptr[B]
 *   kv_pool  bf16 | fp8 [num_slots, 576]
 *   o        bf16 | fp32 [total_q, H, 512]
 *   lse      fp32 [total_q, H]  (natural log)
 *   kv_indptr, qo_indptr int32 [B+1] (non-decreasing), kv_indices int32 [kv_indptr[B]]
 *   Within request b, query row r = t*H + h; rows of one request are contiguous.
 *
 * Conventions.
 *   - The caller owns every buffer.  The library never allocates device memory,
 *     never synchronises and never reads device memory on the host inside
 *     mla_decode_fwd / mla_decode_plan_device / mla_merge_states, so all three
 *     can be captured in a CUDA graph.  `stream` is a cudaStream_t (NULL = the
 *     legacy default stream).
 *   - Every function returns an mla_status and never aborts the process.  Bad
 *     host-visible arguments return MLA_ERR_INVALID_ARG / UNSUPPORTED / ... before
 *     anything is enqueued.  Faults only the device can see (an index outside
 *     [0, num_slots), a decreasing kv_indptr, a plan that does not match the
 *     call, a bounded wait that ran out) are recorded in an error word inside
 *     the workspace; the offending entries are treated as masked.  Read it with
 *     mla_get_device_error.
 *   - Device pointers must be 16-byte aligned (q, kv_pool, o) and 4-byte
 *     aligned (index arrays, lse).
 */
#ifndef MLA_GB300_H
#define MLA_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MLA_ABI_VERSION 6
#define MLA_D_QK 576             /* latent 512 + RoPE 64 */
#define MLA_D_V 512
#define MLA_ROWS_PER_GROUP 256   /* query rows (t,h) of one work item */
#define MLA_BLOCK_N 128          /* KV entries per tile (split granularity) */
#define MLA_MAX_SPLITS 16

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1,
  MLA_ERR_UNSUPPORTED = 2,
  MLA_ERR_WORKSPACE_TOO_SMALL = 3,
  MLA_ERR_PLAN_MISMATCH = 4,
  MLA_ERR_CUDA = 5,
  MLA_ERR_DEVICE_FAULT = 6
} mla_status;

typedef enum { MLA_KV_BF16 = 0, MLA_KV_FP8_E4M3 = 1 } mla_kv_dtype;
typedef enum { MLA_OUT_BF16 = 0, MLA_OUT_FP32 = 1 } mla_out_dtype;
/* Plan modes.
 *   STATIC   built on the host from the query-row counts and a KV capacity
 *            (kv_len_cap) only: one plan serves every call of that shape, so a
 *            captured CUDA graph can replay with any lengths.
 *   DYNAMIC  rebuilt on the device by every mla_decode_fwd from the real
 *            lengths (the persistent-kernel re-plan).
 *   HOST     built on the host by mla_decode_plan from the real kv_indptr and
 *            uploaded by the caller; mla_decode_fwd uses it as is.  Splits and
 *            item order are sized for those lengths.
 * In every mode the forward takes each split's KV range from the lengths it is
 * called with, so a plan never gives a wrong result for other lengths, only a
 * less balanced one. */
typedef enum { MLA_PLAN_STATIC = 0, MLA_PLAN_DYNAMIC = 1, MLA_PLAN_HOST = 2 } mla_plan_mode;

/* Kernel family.  MLA_ALGO_TENSOR (default) is the tcgen05/TMEM kernel;
 * MLA_ALGO_CUDA_CORE is a plain CUDA-core kernel of the same operation, kept for
 * cross-checks.  Both read the same plan and workspace. */
typedef enum { MLA_ALGO_TENSOR = 0, MLA_ALGO_CUDA_CORE = 1 } mla_algo;

/* Device error codes stored in the workspace error word. */
typedef enum {
  MLA_DEV_OK = 0,
  MLA_DEV_BAD_INDEX = 1,        /* kv_indices[j] outside [0, num_slots); info = j        */
  MLA_DEV_BAD_INDPTR = 2,       /* kv_indptr or qo_indptr decreasing; info = b            */
  MLA_DEV_PLAN_MISMATCH = 3,    /* device plan header differs from the call's params     */
  MLA_DEV_ROWS_MISMATCH = 4,    /* q length of request b differs from the plan; info = b */
  MLA_DEV_WAIT_TIMEOUT = 5,     /* a bounded barrier wait ran out; info = site           */
  MLA_DEV_PLAN_OVERFLOW = 6     /* device planner: items exceed the plan capacity        */
} mla_device_error;

/* Plan parameters.  The same struct is passed to the planner and to the forward
 * call; both check the plan against it ("builder and impl call the same
 * predicate").
 *   batch        B >= 0 requests
 *   num_heads    H >= 1
 *   max_q_len    upper bound on T_b (sizes the plan and workspace)
 *   num_workers  W >= 1: the plan aims at about W equal work items' worth of
 *                splitting (use the number of persistent workers)
 *   kv_len_cap   STATIC only: the KV length every request is planned for
 *   mode         mla_plan_mode */
typedef struct {
  int32_t batch;
  int32_t num_heads;
  int32_t max_q_len;
  int32_t num_workers;
  int64_t kv_len_cap;
  int32_t mode;
  int32_t reserved;
} mla_plan_params;

/* Arguments of one forward call.  All pointers are device pointers except
 * `params`, which points to host memory. */
typedef struct {
  const void* q;                     /* bf16 [total_q, H, 576] */
  const void* kv_pool;               /* bf16 | fp8 [num_slots, 576] */
  int64_t num_slots;
  int32_t kv_dtype;                  /* mla_kv_dtype */
  int32_t out_dtype;                 /* mla_out_dtype of o */
  const int32_t* kv_indptr;          /* [B+1] */
  const int32_t* kv_indices;         /* [kv_indptr[B]] */
  const int32_t* qo_indptr;          /* [B+1] */
  int32_t causal;                    /* 0 | 1 */
  int32_t pos_base;                  /* global position of local entry 0 (default 0) */
  int32_t pos_stride;                /* global position step per local entry (>= 1) */
  int32_t algo;                      /* mla_algo */
  const int32_t* pos_base_per_req;   /* nullable [B]: overrides pos_base per request */
  const int32_t* g_kv_indptr;        /* nullable [B+1]: global lengths Lg_b */
  float softmax_scale;               /* finite, > 0 */
  float kv_scale;                    /* fp8: finite, > 0; ignored for bf16 */
  void* o;                           /* [total_q, H, 512] */
  float* lse;                        /* [total_q, H] */
  const mla_plan_params* params;     /* host pointer */
  void* plan_d;                      /* device plan buffer (STATIC: uploaded host plan;
                                        DYNAMIC: rewritten by this call) */
  size_t plan_bytes;
  void* workspace_d;                 /* device workspace, >= the size mla_decode_plan_size gives;
                                        zero-filled once when allocated (since ABI version 6
                                        no call clears it: each completed call leaves its
                                        counters at zero, see mla_get_device_error) */
  size_t ws_bytes;
  /* Index lists that are not a run of positions (since ABI version 3): one index
   * list per layer type -- a sliding window (SWA), a window plus top-k selected
   * entries (CSA), a window plus one compressed entry per 128 tokens (HCA) --
   * over the same decode ("[DSV4] Tuned ASM FP8 decode with split plans; HCA on
   * aiter's persistent V4-NM kernel", Summary part 1). */
  const int32_t* kv_pos;             /* nullable [nnz]: global position of each entry, ascending
                                        within a request; replaces pos_base + i*pos_stride */
  int32_t window;                    /* >= 0; causal only: with W > 0 token t also needs
                                        position > Lg - T + t - W (sliding window); 0 = none */
  int32_t reserved2;                 /* 0 */
} mla_fwd_args;

/* ABI version (MLA_ABI_VERSION); lets a caller probe capabilities by number
 * rather than by inspecting signatures.  3: per-entry positions and the sliding
 * window in mla_fwd_args, HOST plans, mla_cache_write, mla_rope_q_cache;
 * 4: mla_absorb_bmm; 5: work items of 256 query rows over 128-entry tiles (the
 * plan layout changed) and mla_decode_workers; 6: the workspace is zero-filled
 * once by its owner instead of being cleared by every call, and the decode and
 * merge kernels start their set-up while the previous kernel on the stream
 * finishes. */
int mla_abi_version(void);

/* Static description of a status code; never NULL. */
const char* mla_status_string(int status);

/* Number of work items the decode kernel of `algo` (mla_algo) runs at once on
 * the current device: the clusters of the tensor kernel that fit on the GPU
 * together, or the SMs for the CUDA-core kernel.  The persistent workers a plan
 * balances its splits over ("[DSV4] Tuned ASM FP8 decode with split plans; HCA
 * on aiter's persistent V4-NM kernel", Summary part 2); pass it as
 * mla_plan_params.num_workers.  Host call; queries the device's occupancy once
 * per device.  MLA_ERR_INVALID_ARG for an unknown algo or NULL out pointer,
 * MLA_ERR_CUDA if the device cannot be queried. */
mla_status mla_decode_workers(int32_t algo, int32_t* num_workers);

/* Sizes of the plan buffer and of the device workspace for these params.  Both
 * are upper bounds valid for any lengths the params allow.  Host only. */
mla_status mla_decode_plan_size(const mla_plan_params* params, size_t* plan_bytes,
                                size_t* workspace_bytes);

/* Build the plan on the host from host copies of kv_indptr / qo_indptr (each
 * [B+1]; kv_indptr may be NULL in STATIC mode) into plan_h (plan_bytes, host
 * memory).  Pure function of its inputs: the same inputs give the same bytes.
 * Host only; no CUDA call. */
mla_status mla_decode_plan(const mla_plan_params* params, const int32_t* kv_indptr_h,
                           const int32_t* qo_indptr_h, void* plan_h, size_t plan_bytes);

/* The same plan, computed by a kernel from device kv_indptr / qo_indptr and
 * written to plan_d; enqueued on `stream`.  Bit-identical to mla_decode_plan on
 * the same lengths.  Faults go to the workspace error word.  Requires
 * B <= 4096 and an item capacity <= 8192. */
mla_status mla_decode_plan_device(const mla_plan_params* params, const int32_t* kv_indptr_d,
                                  const int32_t* qo_indptr_d, void* plan_d, size_t plan_bytes,
                                  void* workspace_d, size_t ws_bytes, void* stream);

/* Forward call: O and LSE for every (token, head) of the batch.  DYNAMIC mode
 * first re-plans on the device from the real lengths.  Enqueued on `stream`.
 * The decode kernel is launched with programmatic stream serialisation: its
 * set-up (barriers, tensor memory) may run while the kernel before it on the
 * stream finishes, and it reads no input and writes no output before that kernel
 * has completed.  The workspace must have been zero-filled once; the call uses
 * no memset and leaves the workspace's counters at zero when it completes. */
mla_status mla_decode_fwd(const mla_fwd_args* args, void* stream);

/* N-way merge of partial states over disjoint KV subsets:
 *   o_parts [n, rows, dv] (fp32 | bf16, each normalised over its own subset),
 *   lse_parts fp32 [n, rows]  ->  o [rows, dv] (o_dtype), lse fp32 [rows]:
 *   M = max lse_s;  LSE = M + ln sum exp(lse_s - M);  O = sum exp(lse_s - LSE) O_s.
 * States with lse = -inf add nothing; all -inf gives O = 0, LSE = -inf.  This is
 * the combine step of round-robin context parallelism ("Speculative decode +
 * DCP on gfx1250", Problem).  Enqueued on `stream`, with programmatic stream
 * serialisation like mla_decode_fwd: it reads its inputs only after the kernel
 * before it on the stream has completed. */
mla_status mla_merge_states(const void* o_parts, int32_t o_parts_dtype, const float* lse_parts,
                            int32_t n, int64_t rows, int32_t dv, void* o, int32_t o_dtype,
                            float* lse, void* stream);

/* Read and clear the workspace error word.  Synchronises `stream`; not for use
 * while the stream is being captured.  *code receives an mla_device_error and
 * *info its detail; returns MLA_ERR_DEVICE_FAULT when *code != 0.  After a
 * fault it also zeroes the queue words and split counters the faulted call may
 * have left set, so the workspace is ready for the next call. */
mla_status mla_get_device_error(void* workspace_d, void* stream, int32_t* code, int32_t* info);

/* Dtype of an activation input to mla_cache_write. */
typedef enum { MLA_ACT_BF16 = 0, MLA_ACT_FP32 = 1 } mla_act_dtype;

/* Arguments of one KV-cache write.  All pointers are device pointers. */
typedef struct {
  const void* kv_c;             /* [num_tokens, 512] latent columns, rows kv_c_stride elements apart */
  int32_t kv_c_dtype;           /* mla_act_dtype */
  int64_t kv_c_stride;          /* >= 512 */
  const void* k_pe;             /* [num_tokens, 64] RoPE columns, rows k_pe_stride elements apart */
  int32_t k_pe_dtype;           /* mla_act_dtype */
  int64_t k_pe_stride;          /* >= 64 */
  const int32_t* slot_mapping;  /* [num_tokens] pool slot of each token; < 0 = padding */
  int64_t num_tokens;           /* >= 0 */
  void* kv_pool;                /* bf16 | fp8 [num_slots, 576], the pool mla_decode_fwd reads */
  int64_t num_slots;            /* > 0 */
  int32_t kv_dtype;             /* mla_kv_dtype of the pool */
  float kv_scale;               /* fp8: finite, > 0 (stored = value / kv_scale); ignored for bf16 */
} mla_cache_write_args;

/* KV-cache write, the step before the decode: each new token's 512 latent and 64
 * RoPE columns become one 576-wide row of the pool at its slot ("[ROCm] Dspark
 * MLA module", Details: the decode KV-cache write, concat_and_cache_mla, bf16 or
 * fp8 with a per-tensor scale).  For token n with 0 <= slot_mapping[n] < num_slots:
 *   row = (kv_c[n, 0:512], k_pe[n, 0:64]) as float32 (bf16 widens exactly);
 *   bf16 pool: pool[slot] = row rounded to bf16 (nearest, ties to even);
 *   fp8 pool:  pool[slot] = e4m3fn(row * fp32(1/kv_scale)), each product rounded
 *              to float32, then to nearest e4m3fn (ties to even), magnitudes
 *              above 448 saturated to +-448.
 * Tokens with a negative slot (padding) or a slot >= num_slots are skipped.  A
 * slot named twice in one call holds one of the rows (unspecified which).  Each
 * input carries its own dtype and is converted, never reinterpreted: the pages
 * report an fp32 k_pe silently read as bf16 at this step (same page, review
 * comment), so a dtype outside mla_act_dtype is MLA_ERR_INVALID_ARG.  Inputs
 * need 16-byte aligned rows (base pointers 16-byte aligned, strides a multiple
 * of 8 bf16 / 4 fp32 elements), else MLA_ERR_INVALID_ARG.  Enqueued on `stream`;
 * nothing is read back, so the call can be captured in a CUDA graph. */
mla_status mla_cache_write(const mla_cache_write_args* args, void* stream);

/* Rotation layout of the 64 RoPE columns: neox pairs column i with i + 32,
 * interleaved pairs columns 2i and 2i + 1. */
typedef enum { MLA_ROPE_NEOX = 0, MLA_ROPE_INTERLEAVED = 1 } mla_rope_style;

/* Arguments of the fused decode RoPE + q concat + cache write.  Device pointers;
 * every activation is bf16 with 16-byte aligned rows (strides in elements,
 * multiples of 8). */
typedef struct {
  const void* q_nope;              /* [n, H, 512] absorbed latent q */
  int64_t q_nope_stride_token, q_nope_stride_head;
  const void* q_pe;                /* [n, H, 64] RoPE columns of q, not yet rotated */
  int64_t q_pe_stride_token, q_pe_stride_head;
  void* q_out;                     /* [n, H, 576] bf16, contiguous: the q mla_decode_fwd reads */
  int32_t num_heads;               /* H >= 1 */
  int32_t rope_style;              /* mla_rope_style */
  const void* kv_c;                /* [n, 512] */
  int64_t kv_c_stride;             /* >= 512 */
  const void* k_pe;                /* [n, 64], not yet rotated */
  int64_t k_pe_stride;             /* >= 64 */
  const int32_t* positions;        /* [n] position of each token; outside [0, max_pos) clamps */
  const float* cos_sin;            /* fp32 [max_pos, 64]: cos of the 32 angles, then their sin */
  int64_t max_pos;                 /* >= 1 */
  const int32_t* slot_mapping;     /* [n] pool slot; < 0 or >= num_slots: no cache write */
  int64_t num_tokens;              /* n >= 0 */
  void* kv_pool;                   /* bf16 | fp8 [num_slots, 576] */
  int64_t num_slots;
  int32_t kv_dtype;                /* mla_kv_dtype */
  float kv_scale;                  /* fp8: finite, > 0 */
} mla_rope_q_cache_args;

/* Fused decode RoPE + q concat + KV-cache write, the step after the absorb and
 * before the decode ("[ROCm] Dspark MLA module": fused_qk_rope_concat_and_cache_mla,
 * decode RoPE + cache after absorb, a follow-up there).  For token n at position
 * p (clamped), with c = cos_sin[p, 0:32], s = cos_sin[p, 32:64] and the 64 RoPE
 * values split into pairs (a, b) by rope_style:
 *   rotated pair = (a*c - b*s, b*c + a*s), every product and sum rounded to
 *   float32 on its own (no fused multiply-add);
 *   q_out[n, h] = (q_nope[n, h, 0:512], bf16(rotated q_pe[n, h]));
 *   pool[slot_mapping[n]] = the mla_cache_write row of (kv_c[n], rotated k_pe[n]).
 * The rotation runs in float32 and its result is converted for the cache, never
 * reinterpreted (the same page shows a float32 rotated k_pe read as bf16).
 * Enqueued on `stream`; graph-capturable. */
mla_status mla_rope_q_cache(const mla_rope_q_cache_args* args, void* stream);

/* Storage type of an absorb BMM weight. */
typedef enum { MLA_W_BF16 = 0, MLA_W_FP8_E4M3 = 1 } mla_weight_dtype;

/* Arguments of one absorb BMM.  Device pointers; strides in elements. */
typedef struct {
  const void* x;                /* bf16 [num_tokens, num_heads, k], unit stride along k */
  int64_t x_stride_token, x_stride_head;
  const void* w;                /* [num_heads, k, n] contiguous (n fastest): torch.bmm's right operand */
  int32_t w_dtype;              /* mla_weight_dtype */
  float w_scale;                /* per-tensor scale applied to the product; finite (1 for plain bf16) */
  void* out;                    /* bf16 [num_tokens, num_heads, n], unit stride along n */
  int64_t out_stride_token, out_stride_head;
  int32_t num_tokens;           /* >= 0 */
  int32_t num_heads;            /* 1 .. 65535 */
  int32_t k;                    /* multiple of 64, 64 .. 8192 */
  int32_t n;                    /* multiple of 128, 128 .. 8192 */
  int32_t* status_d;            /* optional device int32[2]: a bounded wait that runs out writes
                                   (MLA_DEV_WAIT_TIMEOUT, site); NULL = not recorded */
} mla_absorb_bmm_args;

/* The absorb BMMs either side of the latent decode ("[ROCm] Dspark MLA module",
 * Details: the decode's absorb BMM, an FP8/FP4 BMM when enabled, else torch.bmm):
 * before it q_lat = q_nope @ W_UK per head (k = 128, n = 512), after it
 * out = o_lat @ W_UV per head (k = 512, n = 128).  For every token t and head h:
 *   out[t, h, j] = bf16( w_scale * sum_k x[t, h, k] * w[h, k, j] )
 * with an fp8 weight decoded exactly (e4m3fn), products exact and summed in
 * float32 on the tensor cores, the float32 sum times w_scale rounded to bf16
 * (nearest, ties to even).  The e4m3 NaN codes (0x7F, 0xFF) are outside the
 * contract (they come out finite); sums of signed zeros follow IEEE (-0 + +0 = +0).
 * out may be a column slice of a wider buffer (e.g. the
 * first 512 columns of the 576-wide q) through its strides.  Pointers 16-byte
 * aligned and strides multiples of 8, x_stride_head >= k, out_stride_head >= n,
 * else MLA_ERR_INVALID_ARG.  Enqueued on `stream`; nothing is read back, so the
 * call can be captured in a CUDA graph. */
mla_status mla_absorb_bmm(const mla_absorb_bmm_args* args, void* stream);

/* Forward call for callers that cannot allocate device memory (a runtime or
 * allocator that hands out only input and output tensors): the plan buffer and
 * the workspace come from one static device array of 16 MiB inside the library
 * instead of the caller.  The pages have no counterpart; it is a deployment
 * convenience.  Arguments are those of mla_decode_fwd, except that plan_d,
 * plan_bytes, workspace_d and ws_bytes are ignored.
 *   - DYNAMIC mode only (the plan is rebuilt on the device by every call);
 *     another mode returns MLA_ERR_UNSUPPORTED.
 *   - Problems whose plan plus workspace exceed 16 MiB return
 *     MLA_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *   - Allocates nothing.  The first call on a device looks up that device's
 *     copy of the array (cudaGetSymbolAddress); make it before any stream
 *     capture.  Host threads whose first calls on a device coincide each look
 *     it up and store the same address (an atomic store), so they may race
 *     harmlessly.  The array stays resident while the library is loaded.
 *   - All calls share the array: calls that overlap on the GPU race on it.
 *     Each call clears the state that must start at zero.
 *   - Device-side faults are recorded in the array's error word, which this ABI
 *     does not expose. */
mla_status mla_decode_fwd_noalloc(const mla_fwd_args* args, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MLA_GB300_H */
