/*
 * bsa_fp8.h -- C ABI of the block-sparse FP8 attention prefill library for GB300 (sm_103a).
 *
 * What it computes (Quant Block Sparse Attention, CANNBotDSL sample, section 算子介绍):
 *
 *   Q^_i = Q_i^fp8 * q_descale_i,   K^_j = K_j^fp8 * k_descale_j,   V^_j = V_j^fp8 * v_descale_head(j)
 *   O_i  = sum_{j in A_i} softmax_{j in A_i}( Q^_i . K^_j * softmax_scale ) V^_j
 *   LSE_i = ln sum_{j in A_i} exp( Q^_i . K^_j * softmax_scale )
 *
 * where A_i is the set of keys j of the same sequence that
 *   (1) lie in a 128-token KV tile enabled for the 128-token Q tile of row i -- by a uint8
 *       block_mask (hpc-ops Block-Sparse FP8 Attention, section 块稀疏调度), by a
 *       sparse_indices / sparse_seq_len list (Quant Block Sparse Attention, section
 *       稀疏索引与 PA 页表), or all tiles when neither is given (the dense path);
 *   (2) satisfy j < kv_len (the tail block's padding never takes part);
 *   (3) when causal, satisfy j <= i + (kv_len - q_len)  (right-context causal).
 * A row with an empty A_i gets O_i = 0 and LSE_i = -FLT_MAX.
 *
 * The probabilities are quantised to e4m3 at a fixed scale p_scale (256 by default) before
 * the P.V product and the scale is undone in the epilogue together with the V descale
 * (hpc-ops Block-Sparse FP8 Attention, section 固定 P-scale 量化技巧).
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers of the current CUDA device unless stated.
 *   - The caller owns every buffer.  The library never allocates, frees or synchronises;
 *     all work is queued on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *   - Validation reads only `dims`, scalars and pointer values (null / alignment).  The host
 *     never reads device memory (Quant Block Sparse Attention, section 算子介绍: the host only
 *     checks static parameters and launches asynchronously).
 *   - Errors in device data (a sparse index outside [0, Kb), a sparse_seq_len outside
 *     [0, Kb], a block_table entry outside [0, num_pages) for a needed page, a sequence
 *     length outside its declared maximum) are reported by OR-ing BSA_DEV_* bits into
 *     *dev_status (if dev_status is not NULL) -- read it after synchronising.  The bad
 *     entry is skipped (a bad page reads as zeros); nothing traps or hangs.
 *   - Every wait inside the kernels is bounded (2 s, or bsa_fp8_set_wait_limit_ns); a wait
 *     that runs out sets BSA_DEV_TIMEOUT.
 */
#ifndef BSA_FP8_H
#define BSA_FP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  BSA_OK = 0,
  BSA_ERR_INVALID_ARGUMENT = 1, /* bad dims, scalar, null or misaligned pointer */
  BSA_ERR_UNSUPPORTED = 2,      /* valid but outside what this build supports (GPU arch, Kb,
                                   more than 2^30 (b, h, q-tile) tasks) */
  BSA_ERR_CUDA = 3,             /* a CUDA call or kernel launch failed */
  BSA_ERR_WORKSPACE = 4         /* workspace smaller than bsa_fp8_prefill_workspace_size() */
} bsa_status_t;

/* Quantisation granularity of K and V (hpc-ops article, QuantType list):
 *   QPERTOKEN_PERHEAD_KPERTENSOR_VPERTENSOR      -> k: PER_TENSOR,     v: PER_TENSOR
 *   QPERTOKEN_PERHEAD_KPERTOKEN_PERHEAD_VPERHEAD -> k: PER_TOKEN_HEAD, v: PER_HEAD
 * The second type scales K per token group, head and dimension group.  The only dimension
 * group the pages size is FlashMLA's 1 x 128 tile, which for a 128-wide head is the whole
 * head; a token group's scale is given by repeating it over the group's tokens in the
 * per-token array.  Q is always per token per head. */
typedef enum {
  BSA_SCALE_PER_TENSOR = 0,     /* one fp32 scalar, k_descale[0] / v_descale[0] */
  BSA_SCALE_PER_TOKEN_HEAD = 1, /* K only: fp32 [num_pages, N2, page_size] */
  BSA_SCALE_PER_HEAD = 2        /* V only: fp32 [N2] */
} bsa_scale_kind_t;

/* bits OR-ed into *dev_status */
#define BSA_DEV_BAD_INDEX 1   /* sparse index or sparse_seq_len out of range (entry skipped) */
#define BSA_DEV_BAD_PAGE 2    /* block_table entry out of range for a needed page (reads 0) */
#define BSA_DEV_BAD_SEQLEN 4  /* q_len / kv_len negative or above the declared maximum */
#define BSA_DEV_TIMEOUT 8     /* a bounded wait inside a kernel ran out */

/* Problem geometry (host struct).  Layouts follow the Quant Block Sparse Attention
 * parameter table with the page size made a parameter:
 *   q            e4m3 [total_q, N1, 128]            (TND; row of token t, head h at (t*N1+h)*128)
 *                or [N1, total_q, 128] (NTD) with q_layout = BSA_Q_NTD (the table's layout_q);
 *                q_descale follows: [total_q, N1] or [N1, total_q].  out is always TND.
 *   k/v pages    e4m3 [num_pages, N2, page_size, 128] (HND within a page), or
 *                [num_pages, page_size, N2, 128] (NHD, the hpc-ops tests' other cache layout)
 *                with kv_layout = BSA_KV_NHD.  The per-token K descale stays [num_pages, N2,
 *                page_size] in both.
 *   block_table  int32 [B, max_pages_per_seq]; logical page l of sequence b -> physical page
 * Q tile = KV tile = 128 tokens; Qb = ceil(max_q_len/128), Kb = ceil(max_kv_len/128).
 * The KV head of query head h is h / (N1/N2). */
typedef struct {
  int B;                 /* sequences, >= 0 */
  int N1;                /* query heads, >= 1 */
  int N2;                /* KV heads, N1 % N2 == 0, 1 <= N1/N2 <= 16 */
  int D;                 /* head dim, must be 128 */
  int page_size;         /* tokens per KV page: 32 or 64 */
  int max_q_len;         /* >= every q_len (sets Qb) */
  int max_kv_len;        /* >= every kv_len (sets Kb); Kb <= 4096 */
  int num_pages;         /* physical pages in k/v pages */
  int max_pages_per_seq; /* L, columns of block_table; L * page_size >= max_kv_len */
  int total_q;           /* T = cu_seqlens_q[B] */
  int k_scale_kind;      /* BSA_SCALE_PER_TENSOR or BSA_SCALE_PER_TOKEN_HEAD */
  int v_scale_kind;      /* BSA_SCALE_PER_TENSOR or BSA_SCALE_PER_HEAD */
  int causal;            /* 1 = right-context causal (mask_mode 3), 0 = no causal mask (mode 0) */
  int q_layout;          /* BSA_Q_TND (0) or BSA_Q_NTD (1) */
  int kv_layout;         /* BSA_KV_HND (0) or BSA_KV_NHD (1) */
  int tiles_per_step;    /* active-list tiles per online-softmax step: 1 (or 0) = one 128-token
                            tile; 2 = a 256-wide macro block of two consecutive list tiles, an
                            odd last tile alone (Quant Block Sparse Attention, kernel
                            description): the row maximum that P is quantised against, and the
                            rescale of O, move once per pair.  2 never uses split-KV. */
} bsa_fp8_dims_t;

#define BSA_Q_TND 0
#define BSA_Q_NTD 1
#define BSA_KV_HND 0
#define BSA_KV_NHD 1

/* Bytes of device workspace bsa_fp8_prefill needs for `dims` on the current device: 256 (the
 * counter the persistent kernel's CTAs claim work items from) when every SM pipeline gets a
 * (b, h, q-tile) task; when the tasks cannot occupy half of the pipelines, the prefill cuts
 * each task's active list into up to 8 slices (split-KV) and the workspace also holds, per
 * slice, the un-normalised fp32 O [128, 128] and (m, l) of each row half, plus a counter per
 * task row and half (about 65 KB per slice).  bsa_fp8_prefill zeroes the counters on
 * `stream` before each launch, so two calls in flight at once must not share one workspace;
 * a split plan needs a 256-byte aligned workspace.  Returns 0 for invalid dims;
 * bsa_fp8_prefill reports those. */
size_t bsa_fp8_prefill_workspace_size(const bsa_fp8_dims_t *dims);

/* Block-sparse FP8 attention prefill over a paged KV cache.
 *
 *   q               e4m3 [T, N1, 128], 16-byte aligned
 *   k_pages,v_pages e4m3 [num_pages, N2, page_size, 128], 16-byte aligned; slots past a
 *                   sequence's kv_len in its last page must hold zeros (hpc-ops article,
 *                   快速上手: unused slots are zero-filled)
 *   q_descale       fp32 [T, N1]
 *   k_descale       fp32 [1] (PER_TENSOR) or [num_pages, N2, page_size] (PER_TOKEN_HEAD,
 *                   16-byte aligned)
 *   v_descale       fp32 [1] (PER_TENSOR) or [N2] (PER_HEAD)
 *   cu_seqlens_q    int32 [B+1], cu_seqlens_q[0] = 0, non-decreasing, cu_seqlens_q[B] = T
 *   seqused_kv      int32 [B] KV tokens per sequence, or NULL (then kv_len = q_len)
 *   block_table     int32 [B, max_pages_per_seq]
 *   block_mask      uint8 [B, N1, Qb, Kb], nonzero = compute; or NULL
 *   sparse_indices  int32 [B, N1, Qb, Kb] logical KV tiles per Q tile (any order; only the
 *                   first sparse_seq_len[b,h,qt] entries are read; repeats count once); or NULL
 *   sparse_seq_len  int32 [B, N1, Qb]; required with sparse_indices
 *                   At most one of block_mask / sparse_indices; neither = dense path.
 *   softmax_scale   finite (usually 1/sqrt(128))
 *   p_scale         fixed P-scale; <= 0 selects the default 256; must be finite
 *   out_bf16        bf16 [T, N1, 128] (written), 16-byte aligned
 *   lse_f32         fp32 [N1, T] natural-log LSE (written), 4-byte aligned; or NULL
 *   workspace       device buffer of at least bsa_fp8_prefill_workspace_size(dims) bytes,
 *                   4-byte aligned (BSA_ERR_WORKSPACE otherwise); overwritten by the call
 *   dev_status      device int, OR-ed with BSA_DEV_* bits on data errors; or NULL
 *   stream          cudaStream_t
 */
bsa_status_t bsa_fp8_prefill(const bsa_fp8_dims_t *dims, const void *q, const void *k_pages,
                             const void *v_pages, const float *q_descale, const float *k_descale,
                             const float *v_descale, const int *cu_seqlens_q,
                             const int *seqused_kv, const int *block_table,
                             const uint8_t *block_mask, const int *sparse_indices,
                             const int *sparse_seq_len, float softmax_scale, float p_scale,
                             void *out_bf16, float *lse_f32, void *workspace,
                             size_t workspace_bytes, int *dev_status, void *stream);

/* The active-tile lists the prefill kernel computes, written out so they can be compared
 * bit-exactly (hpc-ops article, section 活跃 tile 列表: a warp ballot writes the active KV
 * tiles of a Q tile in order).  For task (b, h, qt):
 *   tile_lists [B, N1, Qb, Kb] int32: the enabled tiles t < kend(b, qt), ascending, without
 *                                     repeats, then -1 up to Kb
 *   tile_counts [B, N1, Qb] int32:   their number (0 for qt >= ceil(q_len_b/128))
 * kend(b, qt) is the first KV tile no row of the Q tile can see: ceil(min(kv_len,
 * last_row + kv_len - q_len + 1) / 128) when causal, ceil(kv_len / 128) otherwise.
 * Same argument rules and error reporting as bsa_fp8_prefill. */
bsa_status_t bsa_fp8_compact_tiles(const bsa_fp8_dims_t *dims, const int *cu_seqlens_q,
                                   const int *seqused_kv, const uint8_t *block_mask,
                                   const int *sparse_indices, const int *sparse_seq_len,
                                   int *tile_lists, int *tile_counts, int *dev_status,
                                   void *stream);

/* bsa_fp8_prefill without a caller-provided workspace.
 *
 * No counterpart in the pages this library implements: it exists for callers that cannot
 * allocate device memory at the point where they run the prefill -- for example code that
 * only receives the input and output buffers from a host application that owns every
 * allocation (a plugin), code whose device memory comes from a fixed budget reserved at
 * start-up, or code on a path where the implicit synchronisation of cudaMalloc/cudaFree is
 * not acceptable.  This entry point allocates nothing: instead of `workspace` it uses a
 * 256-byte array in the library's own device memory (every GPU that loads the library holds
 * those 256 bytes until the process exits).
 *
 *   - Arguments, layouts, results and errors are exactly those of bsa_fp8_prefill, minus
 *     `workspace` / `workspace_bytes`.  It never uses split-KV, so every valid problem fits
 *     the 256-byte array; a problem for which bsa_fp8_prefill would split runs unsplit here
 *     (the same result up to the rounding of P against each slice's own running max).
 *   - Arguments are checked first, exactly as bsa_fp8_prefill checks them.  Then the first
 *     call on a device (with that device current) looks up the array's device address and
 *     keeps it for later calls; the address is tied to the device's current context and
 *     looked up again after a device reset or a new primary context.  Make that first call
 *     before any stream capture.  A failed lookup returns BSA_ERR_CUDA and leaves no pending
 *     CUDA error.
 *   - Every call on a device shares the one array, which keeps the previous call's contents
 *     (the call clears what must start at zero on `stream` itself).  Calls whose work
 *     overlaps on the GPU -- on different streams without ordering between them -- race on
 *     the array and must not be issued. */
bsa_status_t bsa_fp8_prefill_noalloc(const bsa_fp8_dims_t *dims, const void *q,
                                     const void *k_pages, const void *v_pages,
                                     const float *q_descale, const float *k_descale,
                                     const float *v_descale, const int *cu_seqlens_q,
                                     const int *seqused_kv, const int *block_table,
                                     const uint8_t *block_mask, const int *sparse_indices,
                                     const int *sparse_seq_len, float softmax_scale,
                                     float p_scale, void *out_bf16, float *lse_f32,
                                     int *dev_status, void *stream);

/* The tensors of one prefill call, by the names and layouts bsa_fp8_prefill gives them. */
typedef struct {
  const void *q;
  const void *k_pages;
  const void *v_pages;
  const float *q_descale;
  const float *k_descale;
  const float *v_descale;
  const int *cu_seqlens_q;
  const int *seqused_kv;      /* or NULL */
  const int *block_table;
  const uint8_t *block_mask;  /* or NULL */
  const int *sparse_indices;  /* or NULL */
  const int *sparse_seq_len;  /* or NULL */
  void *out_bf16;
  float *lse_f32;             /* or NULL */
} bsa_fp8_tensors_t;

/* bsa_fp8_prefill on inputs and outputs in HOST memory.
 *
 * `host` holds every tensor in host memory and `dev` a device buffer of the same size for
 * each tensor `host` gives (the optional ones NULL in both, or given in both).  On `stream`
 * the call queues: one host-to-device copy per input tensor (host -> dev), the prefill on
 * the `dev` tensors exactly as bsa_fp8_prefill runs it, then the device-to-host copies of
 * O and, when given, the LSE (dev -> host).  With page-locked host buffers it returns once
 * they are queued; the host outputs are valid after the stream has been synchronised.  Sizes
 * come from `dims`:
 *   q, out            T * N1 * 128 bytes (out: * 2, bf16)
 *   k_pages, v_pages  num_pages * N2 * page_size * 128 bytes
 *   q_descale         T * N1 floats;  lse  N1 * T floats
 *   k_descale         1 float, or num_pages * N2 * page_size (BSA_SCALE_PER_TOKEN_HEAD)
 *   v_descale         1 float, or N2 (BSA_SCALE_PER_HEAD)
 *   cu_seqlens_q      B + 1 ints;  seqused_kv  B ints;  block_table  B * max_pages_per_seq
 *   block_mask        B * N1 * Qb * Kb bytes;  sparse_indices  B * N1 * Qb * Kb ints;
 *   sparse_seq_len    B * N1 * Qb ints
 * Host buffers in page-locked memory (cudaHostAlloc / cudaHostRegister) make the copies
 * asynchronous, so that calls on two streams with separate `dev` sets and workspaces overlap
 * one call's copies with the other's prefill.  Pageable host memory gives the same results,
 * but the CUDA runtime may then hold the calling thread until a copy has completed (for the
 * outputs, until the prefill has finished).
 * Every argument is checked, as bsa_fp8_prefill checks the `dev` set, before anything is
 * queued: BSA_ERR_INVALID_ARGUMENT for a NULL host pointer, a tensor given on one side only,
 * or what bsa_fp8_prefill rejects; BSA_ERR_CUDA if a copy cannot be queued.  `workspace` and
 * `dev_status` are device memory, as for bsa_fp8_prefill.  No counterpart in the pages: the
 * host-to-host path a caller without device buffers of its own inputs runs. */
bsa_status_t bsa_fp8_prefill_host(const bsa_fp8_dims_t *dims, const bsa_fp8_tensors_t *host,
                                  const bsa_fp8_tensors_t *dev, float softmax_scale,
                                  float p_scale, void *workspace, size_t workspace_bytes,
                                  int *dev_status, void *stream);

/* ------------------------------------------------------------------------------------------
 * The quantise step before the attention call: bf16 inputs into the e4m3 + descale format
 * above.  Rule (FlashMLA page, section 量化 / 解量化的源码实现, applied per 128-element row
 * at the granularities the attention pages give): descale = amax / 448 (largest finite
 * e4m3), computed in fp32, or 1 for an all-zero row; code = e4m3(x / descale) with an fp32
 * division, rounded to nearest even and saturated to +-448.  Inputs must be finite.
 * With the UE8M0 rule (the same section's cast of the scale to UE8M0) the descale of a
 * non-zero row is instead the smallest power of two not below amax / 448, so that code times
 * descale is exact; the attention kernels take such descales like any other.
 * ------------------------------------------------------------------------------------------ */

#define BSA_DESCALE_AMAX 0  /* descale = amax / 448 */
#define BSA_DESCALE_UE8M0 1 /* descale = amax / 448 rounded up to a power of two */

/* Quantises `rows` rows of 128 bf16 values (x_bf16 [rows, 128], e.g. Q [T, N1, 128] as
 * rows = T * N1) into codes_e4m3 [rows, 128] and one fp32 descale per row (descale [rows],
 * e.g. q_descale [T, N1]).  x_bf16 and codes_e4m3 must be 16-byte aligned.  rows = 0 is a
 * no-op.  Returns BSA_ERR_INVALID_ARGUMENT for null pointers, misalignment or rows < 0. */
bsa_status_t bsa_fp8_quantize_rows(const void *x_bf16, long long rows, void *codes_e4m3,
                                   float *descale, void *stream);

/* bsa_fp8_quantize_rows under the UE8M0 rule: same arguments, layouts and errors. */
bsa_status_t bsa_fp8_quantize_rows_ue8m0(const void *x_bf16, long long rows, void *codes_e4m3,
                                         float *descale, void *stream);

typedef struct {
  int B;                 /* sequences */
  int N2;                /* KV heads */
  int D;                 /* head dim, must be 128 */
  int page_size;         /* 32 or 64 */
  int num_pages;         /* P */
  int max_pages_per_seq; /* L, columns of block_table */
  int total_new;         /* T_new = cu_seqlens_new[B], rows of k_new / v_new */
  bsa_scale_kind_t k_scale_kind; /* BSA_SCALE_PER_TOKEN_HEAD (computed) or BSA_SCALE_PER_TENSOR */
  bsa_scale_kind_t v_scale_kind; /* BSA_SCALE_PER_HEAD or BSA_SCALE_PER_TENSOR (given) */
  int kv_layout;         /* BSA_KV_HND (0): pages [P, N2, page_size, 128]; BSA_KV_NHD (1):
                            [P, page_size, N2, 128]; k_descale is [P, N2, page_size] in both */
  int k_descale_rule;    /* BSA_DESCALE_AMAX (0) or BSA_DESCALE_UE8M0 (1): the computed
                            per-token K descales (BSA_SCALE_PER_TOKEN_HEAD) */
} bsa_fp8_append_dims_t;

/* Appends new tokens to the paged K/V cache.  Token i of sequence b is row cu_seqlens_new[b]
 * + i of k_new_bf16 / v_new_bf16 [total_new, N2, 128] and lands at logical position
 * pos = cache_seqlens[b] + i: page block_table[b, pos / page_size], slot pos % page_size of
 * k_pages / v_pages (e4m3, HND or NHD pages as dims->kv_layout says).
 *   K, BSA_SCALE_PER_TOKEN_HEAD: each (token, head) row is quantised by the rule above
 *      (UE8M0 when dims->k_descale_rule says so) and
 *      its descale written to k_descale [P, N2, page_size] (k_scale unused, may be NULL).
 *   K, BSA_SCALE_PER_TENSOR: codes = e4m3(x / k_scale[0]) (k_descale unused, may be NULL).
 *   V: codes = e4m3(x / v_scale[head]) for BSA_SCALE_PER_HEAD (v_scale [N2]) or
 *      e4m3(x / v_scale[0]) for BSA_SCALE_PER_TENSOR; the caller chooses the V scale.
 * cu_seqlens_new [B + 1], cache_seqlens [B], block_table [B, L] are device int32.  A token
 * whose page is missing (position beyond L pages, or an entry outside [0, P)) is skipped and
 * BSA_DEV_BAD_PAGE is OR-ed into *dev_status (if given).  Every other slot of the cache is
 * left untouched.  k_new / v_new must be 16-byte aligned.  Counterpart of nothing in the
 * attention pages' interface: it writes their inputs. */
bsa_status_t bsa_fp8_append_kv(const bsa_fp8_append_dims_t *dims, const void *k_new_bf16,
                               const void *v_new_bf16, const int *cu_seqlens_new,
                               const int *cache_seqlens, const int *block_table,
                               const float *k_scale, const float *v_scale, void *k_pages,
                               void *v_pages, float *k_descale, int *dev_status, void *stream);

/* Sets the limit of every bounded wait inside the prefill kernel for launches that follow, in
 * nanoseconds, for the whole process; 0 restores the default of 2 s.  A wait that runs out
 * sets BSA_DEV_TIMEOUT in *dev_status, every role of the CTA stops, waits (with the default
 * limit) for the copies and tensor-core operations it has issued, frees its tensor memory and
 * exits; the results of that launch are then undefined, the CUDA context stays usable.  A
 * watchdog for callers that would rather get an error than wait on a stalled GPU; a limit
 * below the kernel's legitimate waits (microseconds) aborts every launch.  No counterpart in
 * the pages.  Always BSA_OK. */
bsa_status_t bsa_fp8_set_wait_limit_ns(unsigned long long ns);

/* Static text for a status code. */
const char *bsa_status_string(bsa_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* BSA_FP8_H */
