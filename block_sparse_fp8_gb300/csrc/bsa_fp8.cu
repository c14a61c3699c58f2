// Block-sparse FP8 attention prefill over a paged KV cache, for GB300 (sm_103a): host entry
// points of the C ABI (include/bsa_fp8.h) and the exported active-tile list kernel.
//
//   * bsa_compact_kernel -- one warp per (b, h, qt) task writes the ascending list of active
//     KV tiles (warp ballot stream compaction; hpc-ops Block-Sparse FP8 Attention, section
//     活跃 tile 列表).  The attention kernel runs the same device function on its own tasks.
//   * attn::bsa_attention_kernel (bsa_attention.cuh) -- the persistent prefill kernel.
//   * quant::quantize_rows_kernel / quant::append_kv_kernel (bsa_quant.cuh) -- the quantise
//     step that produces the prefill's e4m3 inputs.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "bsa_attention.cuh"
#include "bsa_attention_wide.cuh"
#include "bsa_common.cuh"
#include "bsa_fp8.h"
#include "bsa_quant.cuh"
#include "ptx_sm103.cuh"

namespace bsa {

constexpr int COMPACT_WARPS = 4;

__global__ void __launch_bounds__(COMPACT_WARPS * 32) bsa_compact_kernel(const Params p,
                                                                        int *tile_lists,
                                                                        int *tile_counts) {
  __shared__ uint32_t bitmaps[COMPACT_WARPS][KB_MAX / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long task = (long long)blockIdx.x * COMPACT_WARPS + warp;
  const long long ntasks = (long long)p.B * p.N1 * p.Qb;
  if (task >= ntasks) return;
  const int qt = (int)(task % p.Qb);
  const int h = (int)((task / p.Qb) % p.N1);
  const int b = (int)(task / ((long long)p.Qb * p.N1));
  TaskGeo g = task_geometry(p, b, qt);
  int *list = tile_lists + task * p.Kb;
  int n = compact_task(p, b, h, qt, g.kend, list, bitmaps[warp]);
  for (int t = n + lane; t < p.Kb; t += 32) list[t] = -1;
  if (lane == 0) tile_counts[task] = n;
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

static bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

static int cdiv(long long a, long long b) { return (int)((a + b - 1) / b); }

// Checks only host-visible facts: dims, scalars, pointer nullness and alignment.
static bsa_status_t validate_dims(const bsa_fp8_dims_t *d) {
  if (!d) return BSA_ERR_INVALID_ARGUMENT;
  if (d->D != HEAD_DIM) return BSA_ERR_INVALID_ARGUMENT;
  if (d->page_size != 32 && d->page_size != 64) return BSA_ERR_INVALID_ARGUMENT;
  if (d->B < 0 || d->N1 < 1 || d->N2 < 1 || d->N1 % d->N2 != 0 || d->N1 / d->N2 > 16)
    return BSA_ERR_INVALID_ARGUMENT;
  if (d->max_q_len < 0 || d->max_kv_len < 0 || d->total_q < 0 || d->num_pages < 0 ||
      d->max_pages_per_seq < 0)
    return BSA_ERR_INVALID_ARGUMENT;
  if ((long long)d->max_pages_per_seq * d->page_size < d->max_kv_len)
    return BSA_ERR_INVALID_ARGUMENT;
  if (d->k_scale_kind != BSA_SCALE_PER_TENSOR && d->k_scale_kind != BSA_SCALE_PER_TOKEN_HEAD)
    return BSA_ERR_INVALID_ARGUMENT;
  if (d->v_scale_kind != BSA_SCALE_PER_TENSOR && d->v_scale_kind != BSA_SCALE_PER_HEAD)
    return BSA_ERR_INVALID_ARGUMENT;
  if (d->causal != 0 && d->causal != 1) return BSA_ERR_INVALID_ARGUMENT;
  if (d->q_layout != BSA_Q_TND && d->q_layout != BSA_Q_NTD) return BSA_ERR_INVALID_ARGUMENT;
  if (d->kv_layout != BSA_KV_HND && d->kv_layout != BSA_KV_NHD) return BSA_ERR_INVALID_ARGUMENT;
  if (d->tiles_per_step < 0 || d->tiles_per_step > 2) return BSA_ERR_INVALID_ARGUMENT;
  if (cdiv(d->max_kv_len, TILE) > KB_MAX) return BSA_ERR_UNSUPPORTED;
  // task indices are int; the work-item counter runs past the last task by up to one claim
  // per pipeline, so keep the count well inside int range
  if ((long long)d->B * d->N1 * cdiv(d->max_q_len, TILE) > (1LL << 30))
    return BSA_ERR_UNSUPPORTED;
  return BSA_OK;
}

struct DeviceInfo {
  int state = 0;  // 0 unknown, 1 supported, 2 unsupported
  int num_sms = 0;
  int smem_per_sm = 0;        // shared memory of one SM
  int smem_reserved = 0;      // shared memory the system reserves per resident block
  size_t smem_attr = 0;  // dynamic shared memory the attention kernel is enabled for
  size_t smem_attr_wide = 0;  // ... and the 256-wide macro-block kernel
};

static DeviceInfo g_devices[64];
static std::mutex g_devices_mu;

// sm_103 only; caches the SM count and raises the attention kernel's shared-memory limit.
static bsa_status_t check_device(size_t attn_smem, int *num_sms, int *per_sm = nullptr,
                                 bool wide = false) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
  if (dev < 0 || dev >= 64) return BSA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_devices_mu);
  DeviceInfo &di = g_devices[dev];
  if (di.state == 0) {
    int major = 0, minor = 0, sms = 0, smem_sm = 0, smem_res = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
            cudaSuccess ||
        cudaDeviceGetAttribute(&smem_res, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
            cudaSuccess)
      return BSA_ERR_CUDA;
    di.state = (major == 10 && minor == 3) ? 1 : 2;
    di.num_sms = sms;
    di.smem_per_sm = smem_sm;
    di.smem_reserved = smem_res;
    if (di.state == 1) {
      // The softmax warpgroups raise their registers with setmaxnreg.inc, drawing on what the
      // CTA was launched with; that only completes if the launch allocation covers the
      // whole split, so refuse to launch a build where it does not.
      cudaFuncAttributes fa, fw;
      if (cudaFuncGetAttributes(&fa, attn::bsa_attention_kernel) != cudaSuccess ||
          cudaFuncGetAttributes(&fw, attn_wide::bsa_attention_wide_kernel) != cudaSuccess)
        return BSA_ERR_CUDA;
      if (fa.numRegs * attn::NTHREADS < attn::SPLIT_REGS ||
          fw.numRegs * attn_wide::NTHREADS < attn_wide::SPLIT_REGS)
        di.state = 2;
    }
  }
  if (di.state != 1) return BSA_ERR_UNSUPPORTED;
  size_t &attr = wide ? di.smem_attr_wide : di.smem_attr;
  if (attn_smem > attr) {
    const cudaError_t e =
        wide ? cudaFuncSetAttribute(attn_wide::bsa_attention_wide_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attn_smem)
             : cudaFuncSetAttribute(attn::bsa_attention_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)attn_smem);
    if (e != cudaSuccess) return BSA_ERR_CUDA;
    attr = attn_smem;
  }
  if (num_sms) *num_sms = di.num_sms;
  if (per_sm) *per_sm = 1;  // one CTA per SM: it holds the SM's registers and all of TMEM
  return BSA_OK;
}

// Limit of one bounded wait inside the prefill kernel; 0 selects the default.
static std::atomic<unsigned long long> g_wait_limit_ns{0};

static Params make_params(const bsa_fp8_dims_t *d) {
  Params p;
  memset(&p, 0, sizeof(p));
  const unsigned long long lim = g_wait_limit_ns.load(std::memory_order_relaxed);
  p.wait_limit_ns = lim ? lim : WAIT_LIMIT_NS;
  p.B = d->B;
  p.N1 = d->N1;
  p.N2 = d->N2;
  p.G = d->N1 / d->N2;
  p.ps = d->page_size;
  p.max_q_len = d->max_q_len;
  p.max_kv_len = d->max_kv_len;
  p.num_pages = d->num_pages;
  p.L = d->max_pages_per_seq;
  p.T = d->total_q;
  p.Qb = cdiv(d->max_q_len, TILE);
  p.Kb = cdiv(d->max_kv_len, TILE);
  p.k_per_token = d->k_scale_kind == BSA_SCALE_PER_TOKEN_HEAD;
  p.v_per_head = d->v_scale_kind == BSA_SCALE_PER_HEAD;
  p.causal = d->causal;
  p.q_ntd = d->q_layout == BSA_Q_NTD;
  p.kv_nhd = d->kv_layout == BSA_KV_NHD;
  p.qd_tok = p.q_ntd ? 1 : d->N1;
  p.qd_head = p.q_ntd ? d->total_q : 1;
  return p;
}

static bool encode_map(CUtensorMap *map, const void *base, int rank, const cuuint64_t *dims,
                       const cuuint64_t *strides, const cuuint32_t *box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void *>(base),
                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace bsa

using namespace bsa;

// one int: the work-item counter the persistent CTAs claim work from (padded to 256 bytes)
static constexpr size_t WORKSPACE_BYTES = 256;

namespace {

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Split-KV plan.  When the (b, h, q-tile) tasks cannot occupy half of the pipelines (two per
// SM), each task's active list is cut into S slices (work items) that run on separate
// pipelines and are merged afterwards.  S = min(8, pipelines / tasks, Kb / 16): a slice covers
// at least 16 KV tiles of the task's range.  Splitting costs a partial write and a merge per
// task, which measured more than it saved once every pipeline already had a task.
struct SplitPlan {
  int splits = 1;
  size_t bytes = WORKSPACE_BYTES;           // workspace needed
  size_t off_cnt = 0, off_ml = 0, off_o = 0;
};

SplitPlan plan_splits(const Params &p, int num_sms, bool allow) {
  SplitPlan plan;
  const long long ntasks = (long long)p.B * p.N1 * p.Qb;
  const long long pipes = (long long)attn::NPIPE * std::max(num_sms, 1);
  if (!allow || ntasks <= 0 || 2 * ntasks > pipes) return plan;
  const int best = (int)std::min<long long>(std::min<long long>(attn::MAX_SPLITS, pipes / ntasks),
                                             p.Kb / 16);
  if (best <= 1) return plan;
  const long long items = ntasks * best;
  plan.splits = best;
  plan.off_cnt = WORKSPACE_BYTES;
  plan.off_ml = plan.off_cnt + round256((size_t)ntasks * TILE * 2 * sizeof(int));
  plan.off_o = plan.off_ml + round256((size_t)items * TILE * 2 * 2 * sizeof(float));
  plan.bytes = plan.off_o + (size_t)items * TILE * HEAD_DIM * sizeof(float);
  return plan;
}

}  // namespace

extern "C" size_t bsa_fp8_prefill_workspace_size(const bsa_fp8_dims_t *dims) {
  if (validate_dims(dims) != BSA_OK) return 0;
  int num_sms = 0;
  if (check_device(0, &num_sms) != BSA_OK) return WORKSPACE_BYTES;
  return plan_splits(make_params(dims), num_sms, dims->tiles_per_step != 2).bytes;
}

extern "C" bsa_status_t bsa_fp8_set_wait_limit_ns(unsigned long long ns) {
  g_wait_limit_ns.store(ns, std::memory_order_relaxed);
  return BSA_OK;
}

extern "C" const char *bsa_status_string(bsa_status_t status) {
  switch (status) {
    case BSA_OK: return "ok";
    case BSA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case BSA_ERR_UNSUPPORTED: return "unsupported (device or size)";
    case BSA_ERR_CUDA: return "CUDA error";
    case BSA_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

extern "C" bsa_status_t bsa_fp8_compact_tiles(const bsa_fp8_dims_t *dims, const int *cu_seqlens_q,
                                              const int *seqused_kv, const uint8_t *block_mask,
                                              const int *sparse_indices,
                                              const int *sparse_seq_len, int *tile_lists,
                                              int *tile_counts, int *dev_status, void *stream) {
  bsa_status_t st = validate_dims(dims);
  if (st != BSA_OK) return st;
  if (block_mask && sparse_indices) return BSA_ERR_INVALID_ARGUMENT;
  if (sparse_indices && !sparse_seq_len) return BSA_ERR_INVALID_ARGUMENT;
  Params p = make_params(dims);
  const long long ntasks = (long long)p.B * p.N1 * p.Qb;
  if (ntasks == 0 || p.Kb == 0) return BSA_OK;
  if (!cu_seqlens_q || !tile_lists || !tile_counts) return BSA_ERR_INVALID_ARGUMENT;
  st = check_device(0, nullptr);
  if (st != BSA_OK) return st;
  p.cu_seqlens_q = cu_seqlens_q;
  p.seqused_kv = seqused_kv;
  p.block_mask = block_mask;
  p.sparse_indices = sparse_indices;
  p.sparse_seq_len = sparse_seq_len;
  p.dev_status = dev_status;
  const long long blocks = (ntasks + COMPACT_WARPS - 1) / COMPACT_WARPS;
  bsa_compact_kernel<<<(unsigned)blocks, COMPACT_WARPS * 32, 0, (cudaStream_t)stream>>>(
      p, tile_lists, tile_counts);
  return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

// ------------------------------------------------------------------------------------------
// The workspace of bsa_fp8_prefill_noalloc, for callers that cannot allocate device memory:
// this file-scope array, 256 bytes on every device that loads the library.
// ------------------------------------------------------------------------------------------

namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = 256;
static_assert(NOALLOC_SCRATCH_BYTES >= WORKSPACE_BYTES,
              "the array must hold the unsplit prefill's workspace");
static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

// Host code cannot pass g_noalloc_scratch itself to a kernel (on the host that name is only a
// stand-in for the device symbol): look up the device address with the device current and
// reuse it.  The address belongs to the context the module was loaded into, so it is cached
// together with that context's ID and looked up again when the ID changes (a device reset or
// a recreated primary context loads the module afresh, possibly at another address).
struct NoallocAddr {
  unsigned long long ctx_id = 0;
  void *ptr = nullptr;
};
NoallocAddr g_noalloc_addr[64];
std::mutex g_noalloc_mu;

struct CtxFns {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxFns &ctx_fns() {
  static CtxFns fns;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
    ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fns.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(ptr);
  });
  return fns;
}

// Called after check_device(), so the device's primary context is current.
bsa_status_t noalloc_scratch(void **addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
  if (dev < 0 || dev >= 64) return BSA_ERR_UNSUPPORTED;
  const CtxFns &fns = ctx_fns();
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!fns.get_current || !fns.get_id || fns.get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      fns.get_id(ctx, &id) != CUDA_SUCCESS)
    return BSA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocAddr &a = g_noalloc_addr[dev];
  if (!a.ptr || a.ctx_id != id) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      (void)cudaGetLastError();  // leave no pending error behind for the caller
      return BSA_ERR_CUDA;
    }
    a.ptr = ptr;
    a.ctx_id = id;
  }
  *addr = a.ptr;
  return BSA_OK;
}

}  // namespace

// The prefill.  With `noalloc` it ignores workspace / workspace_bytes and uses the library's
// own array instead (never split-KV); otherwise the caller's workspace must hold the split
// plan's bytes.  With `check_only` it returns after every check (the tensor maps' encoding
// included), before anything is queued.
static bsa_status_t prefill_impl(const bsa_fp8_dims_t *dims, const void *q, const void *k_pages,
                                 const void *v_pages, const float *q_descale,
                                 const float *k_descale, const float *v_descale,
                                 const int *cu_seqlens_q, const int *seqused_kv,
                                 const int *block_table, const uint8_t *block_mask,
                                 const int *sparse_indices, const int *sparse_seq_len,
                                 float softmax_scale, float p_scale, void *out_bf16,
                                 float *lse_f32, void *workspace, size_t workspace_bytes,
                                 int *dev_status, void *stream, bool noalloc,
                                 bool check_only = false) {
  bsa_status_t st = validate_dims(dims);
  if (st != BSA_OK) return st;
  if (block_mask && sparse_indices) return BSA_ERR_INVALID_ARGUMENT;
  if (sparse_indices && !sparse_seq_len) return BSA_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(softmax_scale)) return BSA_ERR_INVALID_ARGUMENT;
  if (std::isnan(p_scale) || std::isinf(p_scale)) return BSA_ERR_INVALID_ARGUMENT;
  if (p_scale <= 0.f) p_scale = 256.f;
  Params p = make_params(dims);
  const long long ntasks = (long long)p.B * p.N1 * p.Qb;
  if (ntasks == 0 || p.T == 0) return BSA_OK;
  if (!q || !k_pages || !v_pages || !q_descale || !k_descale || !v_descale || !cu_seqlens_q ||
      !block_table || !out_bf16)
    return BSA_ERR_INVALID_ARGUMENT;
  if (p.num_pages < 1 || p.L < 1) return BSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) ||
      (p.k_per_token && !aligned16(k_descale)) || !aligned16(out_bf16) ||
      (reinterpret_cast<uintptr_t>(lse_f32) & 3u) != 0)
    return BSA_ERR_INVALID_ARGUMENT;
  if (!noalloc && (!workspace || workspace_bytes < WORKSPACE_BYTES ||
                   (reinterpret_cast<uintptr_t>(workspace) & 3u) != 0))
    return BSA_ERR_WORKSPACE;
  // 256-wide macro blocks (two list tiles per online-softmax step) run their own kernel
  const bool wide = dims->tiles_per_step == 2;
  const size_t smem = wide ? attn_wide::smem_bytes(p.Kb) : attn::smem_bytes(p.Kb);
  int num_sms = 0, per_sm = 1;
  st = check_device(smem, &num_sms, &per_sm, wide);
  if (st != BSA_OK) return st;
  if (noalloc) {
    // the library's own array, looked up only once every argument has been checked
    st = noalloc_scratch(&workspace);
    if (st != BSA_OK) return st;
    workspace_bytes = NOALLOC_SCRATCH_BYTES;
  }
  // the array-backed entry point never splits: its array holds the item counter only; nor do
  // macro blocks (a slice boundary would cut a pair)
  const SplitPlan plan = plan_splits(p, num_sms, !noalloc && !wide);
  if (workspace_bytes < plan.bytes ||
      (plan.splits > 1 && (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
    return BSA_ERR_WORKSPACE;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  p.splits = plan.splits;
  if (plan.splits > 1) {
    p.row_cnt = reinterpret_cast<int *>(ws + plan.off_cnt);
    p.part_ml = reinterpret_cast<float *>(ws + plan.off_ml);
    p.part_o = reinterpret_cast<float *>(ws + plan.off_o);
  }

  p.q_descale = q_descale;
  p.k_descale = k_descale;
  p.v_descale = v_descale;
  p.cu_seqlens_q = cu_seqlens_q;
  p.seqused_kv = seqused_kv;
  p.block_table = block_table;
  p.block_mask = block_mask;
  p.sparse_indices = sparse_indices;
  p.sparse_seq_len = sparse_seq_len;
  p.out = static_cast<__nv_bfloat16 *>(out_bf16);
  p.lse = lse_f32;
  p.dev_status = dev_status;
  p.task_counter = static_cast<int *>(workspace);
  p.scale_log2 = (float)((double)softmax_scale * 1.4426950408889634);
  p.log2_pscale = (float)std::log2((double)p_scale);
  p.ln_pscale = (float)std::log((double)p_scale);

  // Tensor maps, innermost dimension first.  Either layout puts one 128-token Q box of a head,
  // or one page of a KV head, into shared memory as consecutive 128-byte rows.
  CUtensorMap tq, tk, tv;
  if (!p.q_ntd) {  // [T, N1, 128]: dims (d, head, token), box (128, 1, 128)
    cuuint64_t gd[3] = {HEAD_DIM, (cuuint64_t)p.N1, (cuuint64_t)p.T};
    cuuint64_t gs[2] = {HEAD_DIM, (cuuint64_t)p.N1 * HEAD_DIM};
    cuuint32_t box[3] = {HEAD_DIM, 1, TILE};
    if (!encode_map(&tq, q, 3, gd, gs, box)) return BSA_ERR_CUDA;
  } else {         // [N1, T, 128]: dims (d, token, head), box (128, 128, 1)
    cuuint64_t gd[3] = {HEAD_DIM, (cuuint64_t)p.T, (cuuint64_t)p.N1};
    cuuint64_t gs[2] = {HEAD_DIM, (cuuint64_t)p.T * HEAD_DIM};
    cuuint32_t box[3] = {HEAD_DIM, TILE, 1};
    if (!encode_map(&tq, q, 3, gd, gs, box)) return BSA_ERR_CUDA;
  }
  if (!p.kv_nhd) {  // [P, N2, ps, 128]: dims (d, slot, head, page), box (128, ps, 1, 1)
    cuuint64_t gd[4] = {HEAD_DIM, (cuuint64_t)p.ps, (cuuint64_t)p.N2, (cuuint64_t)p.num_pages};
    cuuint64_t gs[3] = {HEAD_DIM, (cuuint64_t)p.ps * HEAD_DIM,
                        (cuuint64_t)p.N2 * p.ps * HEAD_DIM};
    cuuint32_t box[4] = {HEAD_DIM, (cuuint32_t)p.ps, 1, 1};
    if (!encode_map(&tk, k_pages, 4, gd, gs, box)) return BSA_ERR_CUDA;
    if (!encode_map(&tv, v_pages, 4, gd, gs, box)) return BSA_ERR_CUDA;
  } else {          // [P, ps, N2, 128]: dims (d, head, slot, page), box (128, 1, ps, 1)
    cuuint64_t gd[4] = {HEAD_DIM, (cuuint64_t)p.N2, (cuuint64_t)p.ps, (cuuint64_t)p.num_pages};
    cuuint64_t gs[3] = {HEAD_DIM, (cuuint64_t)p.N2 * HEAD_DIM,
                        (cuuint64_t)p.ps * p.N2 * HEAD_DIM};
    cuuint32_t box[4] = {HEAD_DIM, 1, (cuuint32_t)p.ps, 1};
    if (!encode_map(&tk, k_pages, 4, gd, gs, box)) return BSA_ERR_CUDA;
    if (!encode_map(&tv, v_pages, 4, gd, gs, box)) return BSA_ERR_CUDA;
  }
  if (check_only) return BSA_OK;  // every check done, the tensor maps included
  // persistent grid: one CTA per SM (two pipelines each)
  const long long items = ntasks * plan.splits;
  const long long grid = std::min<long long>(items, (long long)per_sm * num_sms);
  // the item counter, and with split-KV the per-row completion counters, start at zero
  const size_t zero_bytes = plan.splits > 1 ? plan.off_ml : sizeof(int);
  if (cudaMemsetAsync(workspace, 0, zero_bytes, (cudaStream_t)stream) != cudaSuccess)
    return BSA_ERR_CUDA;
  if (wide)
    attn_wide::bsa_attention_wide_kernel<<<(unsigned)grid, attn_wide::NTHREADS, smem,
                                           (cudaStream_t)stream>>>(p, tq, tk, tv);
  else
    attn::bsa_attention_kernel<<<(unsigned)grid, attn::NTHREADS, smem, (cudaStream_t)stream>>>(
        p, tq, tk, tv);
  return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

extern "C" bsa_status_t bsa_fp8_prefill(const bsa_fp8_dims_t *dims, const void *q,
                                        const void *k_pages, const void *v_pages,
                                        const float *q_descale, const float *k_descale,
                                        const float *v_descale, const int *cu_seqlens_q,
                                        const int *seqused_kv, const int *block_table,
                                        const uint8_t *block_mask, const int *sparse_indices,
                                        const int *sparse_seq_len, float softmax_scale,
                                        float p_scale, void *out_bf16, float *lse_f32,
                                        void *workspace, size_t workspace_bytes,
                                        int *dev_status, void *stream) {
  return prefill_impl(dims, q, k_pages, v_pages, q_descale, k_descale, v_descale, cu_seqlens_q,
                      seqused_kv, block_table, block_mask, sparse_indices, sparse_seq_len,
                      softmax_scale, p_scale, out_bf16, lse_f32, workspace, workspace_bytes,
                      dev_status, stream, false);
}

extern "C" bsa_status_t bsa_fp8_prefill_host(const bsa_fp8_dims_t *dims,
                                             const bsa_fp8_tensors_t *host,
                                             const bsa_fp8_tensors_t *dev, float softmax_scale,
                                             float p_scale, void *workspace,
                                             size_t workspace_bytes, int *dev_status,
                                             void *stream) {
  if (!host || !dev) return BSA_ERR_INVALID_ARGUMENT;
  bsa_status_t st = validate_dims(dims);
  if (st != BSA_OK) return st;
  const Params p = make_params(dims);
  // an empty problem queues nothing, as bsa_fp8_prefill launches nothing for it
  const bool empty = (long long)p.B * p.N1 * p.Qb == 0 || p.T == 0;
  // every tensor of the device set has its host counterpart, and the reverse
  if (!empty && (!host->q || !host->k_pages || !host->v_pages || !host->q_descale ||
                 !host->k_descale || !host->v_descale || !host->cu_seqlens_q ||
                 !host->block_table || !host->out_bf16))
    return BSA_ERR_INVALID_ARGUMENT;
  if (!empty && (!host->seqused_kv != !dev->seqused_kv || !host->block_mask != !dev->block_mask ||
                 !host->sparse_indices != !dev->sparse_indices ||
                 !host->sparse_seq_len != !dev->sparse_seq_len || !host->lse_f32 != !dev->lse_f32))
    return BSA_ERR_INVALID_ARGUMENT;
  const auto run = [&](bool check_only) {
    return prefill_impl(dims, dev->q, dev->k_pages, dev->v_pages, dev->q_descale,
                        dev->k_descale, dev->v_descale, dev->cu_seqlens_q, dev->seqused_kv,
                        dev->block_table, dev->block_mask, dev->sparse_indices,
                        dev->sparse_seq_len, softmax_scale, p_scale, dev->out_bf16,
                        dev->lse_f32, workspace, workspace_bytes, dev_status, stream, false,
                        check_only);
  };
  st = run(true);
  if (st != BSA_OK || empty) return st;

  const size_t T = (size_t)p.T, N1 = (size_t)p.N1, N2 = (size_t)p.N2, B = (size_t)p.B;
  const size_t cache_rows = (size_t)p.num_pages * N2 * (size_t)p.ps;
  const size_t tasks = B * N1 * (size_t)p.Qb;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const auto copy = [&](const void *dst, const void *src, size_t bytes, cudaMemcpyKind kind) {
    if (!src || bytes == 0) return true;
    if (cudaMemcpyAsync(const_cast<void *>(dst), src, bytes, kind, s) == cudaSuccess) return true;
    cudaGetLastError();  // leave no pending error behind
    return false;
  };
  const cudaMemcpyKind in = cudaMemcpyHostToDevice;
  const bool queued =
      copy(dev->q, host->q, T * N1 * HEAD_DIM, in) &&
      copy(dev->k_pages, host->k_pages, cache_rows * HEAD_DIM, in) &&
      copy(dev->v_pages, host->v_pages, cache_rows * HEAD_DIM, in) &&
      copy(dev->q_descale, host->q_descale, T * N1 * sizeof(float), in) &&
      copy(dev->k_descale, host->k_descale, (p.k_per_token ? cache_rows : 1) * sizeof(float),
           in) &&
      copy(dev->v_descale, host->v_descale, (p.v_per_head ? N2 : 1) * sizeof(float), in) &&
      copy(dev->cu_seqlens_q, host->cu_seqlens_q, (B + 1) * sizeof(int), in) &&
      copy(dev->seqused_kv, host->seqused_kv, B * sizeof(int), in) &&
      copy(dev->block_table, host->block_table, B * (size_t)p.L * sizeof(int), in) &&
      copy(dev->block_mask, host->block_mask, tasks * (size_t)p.Kb, in) &&
      copy(dev->sparse_indices, host->sparse_indices, tasks * (size_t)p.Kb * sizeof(int), in) &&
      copy(dev->sparse_seq_len, host->sparse_seq_len, tasks * sizeof(int), in);
  if (!queued) return BSA_ERR_CUDA;
  st = run(false);
  if (st != BSA_OK) return st;
  const cudaMemcpyKind out = cudaMemcpyDeviceToHost;
  if (!copy(host->out_bf16, dev->out_bf16, T * N1 * HEAD_DIM * 2, out) ||
      !copy(host->lse_f32, dev->lse_f32, N1 * T * sizeof(float), out))
    return BSA_ERR_CUDA;
  return BSA_OK;
}

// ------------------------------------------------------------------------------------------
// quantise step
// ------------------------------------------------------------------------------------------

namespace {

// grid for `rows` half-warp rows (two per half-warp step): enough blocks to cover them, at
// most as many as are resident at once
template <typename Kernel>
bsa_status_t quant_grid(Kernel kernel, long long rows, unsigned *grid) {
  int num_sms = 0, per_sm = 0;
  const bsa_status_t st = check_device(0, &num_sms);
  if (st != BSA_OK) return st;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, quant::THREADS, 0) !=
      cudaSuccess)
    return BSA_ERR_CUDA;
  const long long per_block = 2 * (quant::THREADS / 16);
  const long long need = (rows + per_block - 1) / per_block;
  *grid = (unsigned)std::max<long long>(
      1, std::min<long long>(need, (long long)std::max(per_sm, 1) * num_sms));
  return BSA_OK;
}

}  // namespace

static bsa_status_t quantize_rows_impl(const void *x_bf16, long long rows, void *codes_e4m3,
                                       float *descale, void *stream, bool ue8m0) {
  if (rows < 0) return BSA_ERR_INVALID_ARGUMENT;
  if (rows == 0) return BSA_OK;
  if (!x_bf16 || !codes_e4m3 || !descale || !aligned16(x_bf16) || !aligned16(codes_e4m3))
    return BSA_ERR_INVALID_ARGUMENT;
  unsigned grid = 0;
  const bsa_status_t st = quant_grid(quant::quantize_rows_kernel, rows, &grid);
  if (st != BSA_OK) return st;
  quant::quantize_rows_kernel<<<grid, quant::THREADS, 0, (cudaStream_t)stream>>>(
      static_cast<const uint4 *>(x_bf16), rows, static_cast<uint2 *>(codes_e4m3), descale,
      ue8m0);
  return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

extern "C" bsa_status_t bsa_fp8_quantize_rows(const void *x_bf16, long long rows,
                                              void *codes_e4m3, float *descale, void *stream) {
  return quantize_rows_impl(x_bf16, rows, codes_e4m3, descale, stream, false);
}

extern "C" bsa_status_t bsa_fp8_quantize_rows_ue8m0(const void *x_bf16, long long rows,
                                                    void *codes_e4m3, float *descale,
                                                    void *stream) {
  return quantize_rows_impl(x_bf16, rows, codes_e4m3, descale, stream, true);
}

extern "C" bsa_status_t bsa_fp8_append_kv(const bsa_fp8_append_dims_t *d, const void *k_new_bf16,
                                          const void *v_new_bf16, const int *cu_seqlens_new,
                                          const int *cache_seqlens, const int *block_table,
                                          const float *k_scale, const float *v_scale,
                                          void *k_pages, void *v_pages, float *k_descale,
                                          int *dev_status, void *stream) {
  if (!d || d->D != HEAD_DIM || (d->page_size != 32 && d->page_size != 64) || d->B < 0 ||
      d->N2 < 1 || d->num_pages < 0 || d->max_pages_per_seq < 0 || d->total_new < 0)
    return BSA_ERR_INVALID_ARGUMENT;
  if (d->k_scale_kind != BSA_SCALE_PER_TOKEN_HEAD && d->k_scale_kind != BSA_SCALE_PER_TENSOR)
    return BSA_ERR_INVALID_ARGUMENT;
  if (d->v_scale_kind != BSA_SCALE_PER_HEAD && d->v_scale_kind != BSA_SCALE_PER_TENSOR)
    return BSA_ERR_INVALID_ARGUMENT;
  if (d->kv_layout != BSA_KV_HND && d->kv_layout != BSA_KV_NHD) return BSA_ERR_INVALID_ARGUMENT;
  if (d->k_descale_rule != BSA_DESCALE_AMAX && d->k_descale_rule != BSA_DESCALE_UE8M0)
    return BSA_ERR_INVALID_ARGUMENT;
  const long long rows = (long long)d->total_new * d->N2;
  if (rows == 0 || d->B == 0) return BSA_OK;
  const bool k_tok = d->k_scale_kind == BSA_SCALE_PER_TOKEN_HEAD;
  if (!k_new_bf16 || !v_new_bf16 || !cu_seqlens_new || !cache_seqlens || !block_table ||
      !v_scale || !k_pages || !v_pages || (k_tok ? !k_descale : !k_scale))
    return BSA_ERR_INVALID_ARGUMENT;
  if (!aligned16(k_new_bf16) || !aligned16(v_new_bf16) || !aligned16(k_pages) ||
      !aligned16(v_pages))
    return BSA_ERR_INVALID_ARGUMENT;
  unsigned grid = 0;
  const bsa_status_t st = quant_grid(quant::append_kv_kernel, rows, &grid);
  if (st != BSA_OK) return st;
  quant::AppendParams p;
  p.k_new = static_cast<const uint4 *>(k_new_bf16);
  p.v_new = static_cast<const uint4 *>(v_new_bf16);
  p.cu_new = cu_seqlens_new;
  p.cache_len = cache_seqlens;
  p.block_table = block_table;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.k_pages = static_cast<uint2 *>(k_pages);
  p.v_pages = static_cast<uint2 *>(v_pages);
  p.k_descale = k_descale;
  p.dev_status = dev_status;
  p.B = d->B;
  p.N2 = d->N2;
  p.ps = d->page_size;
  p.num_pages = d->num_pages;
  p.L = d->max_pages_per_seq;
  p.total_new = d->total_new;
  p.k_per_token = k_tok ? 1 : 0;
  p.v_per_head = d->v_scale_kind == BSA_SCALE_PER_HEAD ? 1 : 0;
  p.kv_nhd = d->kv_layout == BSA_KV_NHD ? 1 : 0;
  p.k_ue8m0 = d->k_descale_rule == BSA_DESCALE_UE8M0 ? 1 : 0;
  quant::append_kv_kernel<<<grid, quant::THREADS, 0, (cudaStream_t)stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}

extern "C" bsa_status_t bsa_fp8_prefill_noalloc(
    const bsa_fp8_dims_t *dims, const void *q, const void *k_pages, const void *v_pages,
    const float *q_descale, const float *k_descale, const float *v_descale,
    const int *cu_seqlens_q, const int *seqused_kv, const int *block_table,
    const uint8_t *block_mask, const int *sparse_indices, const int *sparse_seq_len,
    float softmax_scale, float p_scale, void *out_bf16, float *lse_f32, int *dev_status,
    void *stream) {
  // every argument is checked as bsa_fp8_prefill checks it; the array is looked up after that
  return prefill_impl(dims, q, k_pages, v_pages, q_descale, k_descale, v_descale, cu_seqlens_q,
                      seqused_kv, block_table, block_mask, sparse_indices, sparse_seq_len,
                      softmax_scale, p_scale, out_bf16, lse_f32, nullptr, 0, dev_status, stream,
                      true);
}
