// Shared device code: kernel parameters, task geometry and the active-tile compaction that
// both the exported list kernel and the attention kernel run.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "bsa_fp8.h"

namespace bsa {

constexpr int TILE = 128;
constexpr int HEAD_DIM = 128;
constexpr int KB_MAX = 4096;
// Default limit of a bounded wait inside the kernels (2 s: far above any legitimate wait); the
// host may lower it for a launch (Params::wait_limit_ns).  Draining in-flight copies after an
// abort always uses this default.
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;

struct Params {
  const float *q_descale;
  const float *k_descale;
  const float *v_descale;
  const int *cu_seqlens_q;
  const int *seqused_kv;
  const int *block_table;
  const uint8_t *block_mask;
  const int *sparse_indices;
  const int *sparse_seq_len;
  __nv_bfloat16 *out;
  float *lse;
  int *dev_status;
  int *task_counter;  // zeroed before launch; CTAs claim work-item indices from it
  // split-KV (splits > 1): per work item and row, the un-normalised O (fp32 [item][128][128])
  // and (m, l) per row half ([item][128][2] float2); per task, row and half a counter of the
  // items done (zeroed before launch)
  int splits;
  float *part_o;
  float *part_ml;
  int *row_cnt;
  int B, N1, N2, G, ps, max_q_len, max_kv_len, num_pages, L, T, Qb, Kb;
  int k_per_token, v_per_head, causal;
  int q_ntd, kv_nhd;  // layouts: Q [N1, T, 128] (q_descale [N1, T]); pages [P, ps, N2, 128]
  int qd_tok, qd_head;  // q_descale element strides of a token and of a head
  unsigned long long wait_limit_ns;  // a wait that runs longer aborts the launch
  float scale_log2;   // softmax_scale * log2(e)
  float log2_pscale;  // log2(p_scale)
  float ln_pscale;    // ln(p_scale)
};

__device__ __forceinline__ void report(const Params &p, int bits) {
  if (p.dev_status) atomicOr(p.dev_status, bits);
}

// Sequence geometry of task (b, qt).  kend = first KV tile that no row of the Q tile can see.
struct TaskGeo {
  int q0, q_len, kv_len, kend;
  bool valid;
};

__device__ __forceinline__ TaskGeo task_geometry(const Params &p, int b, int qt) {
  TaskGeo g;
  int c0 = p.cu_seqlens_q[b], c1 = p.cu_seqlens_q[b + 1];
  int ql = c1 - c0;
  int kl = p.seqused_kv ? p.seqused_kv[b] : ql;
  bool bad = c0 < 0 || ql < 0 || ql > p.max_q_len || c1 > p.T || kl < 0 || kl > p.max_kv_len ||
             (long long)kl > (long long)p.L * p.ps;
  if (bad) {
    report(p, BSA_DEV_BAD_SEQLEN);
    ql = 0;
    kl = 0;
  }
  g.q0 = c0;
  g.q_len = ql;
  g.kv_len = kl;
  g.valid = qt * TILE < ql;
  int lim = kl;
  if (p.causal) {
    int last_row = min(qt * TILE + TILE, ql) - 1;
    lim = min(lim, last_row + (kl - ql) + 1);
  }
  lim = max(lim, 0);
  g.kend = g.valid ? min((lim + TILE - 1) / TILE, p.Kb) : 0;
  return g;
}

// Warp-cooperative active-tile compaction for task (b, h, qt): the enabled tiles t < kend,
// ascending, without repeats (hpc-ops Block-Sparse FP8 Attention, section 活跃 tile 列表: one
// warp ballot writes the active KV tiles of a Q tile in order).  `bitmap` is KB_MAX/32 words
// of this warp's shared memory (used by the index-list form).  Returns the count.
template <typename OutT>
__device__ int compact_task(const Params &p, int b, int h, int qt, int kend, OutT *list,
                            uint32_t *bitmap) {
  const int lane = threadIdx.x & 31;
  const size_t task = ((size_t)b * p.N1 + h) * p.Qb + qt;
  const size_t row = task * (size_t)p.Kb;
  int n = 0;
  if (p.block_mask) {
    for (int base = 0; base < kend; base += 32) {
      int t = base + lane;
      bool on = t < kend && p.block_mask[row + t] != 0;
      unsigned bal = __ballot_sync(0xffffffffu, on);
      if (on) list[n + __popc(bal & ((1u << lane) - 1u))] = static_cast<OutT>(t);
      n += __popc(bal);
    }
  } else if (p.sparse_indices) {
    // the first 32 entries of the row are read together with its length (they lie inside the
    // [B, N1, Qb, Kb] row whatever the length), so a list of up to 32 entries costs one round
    // trip to memory instead of two
    const int first = lane < p.Kb ? p.sparse_indices[row + lane] : -1;
    int len = p.sparse_seq_len[task];
    if (len < 0 || len > p.Kb) {
      if (lane == 0) report(p, BSA_DEV_BAD_INDEX);
      len = len < 0 ? 0 : p.Kb;
    }
    const int nwords = (kend + 31) >> 5;
    for (int w = lane; w < nwords; w += 32) bitmap[w] = 0u;
    __syncwarp();
    for (int e = lane; e < len; e += 32) {
      const int t = e < 32 ? first : p.sparse_indices[row + e];
      if (t < 0 || t >= p.Kb)
        report(p, BSA_DEV_BAD_INDEX);
      else if (t < kend)
        atomicOr(&bitmap[t >> 5], 1u << (t & 31));
    }
    __syncwarp();
    for (int base = 0; base < kend; base += 32) {
      bool on = base + lane < kend && ((bitmap[base >> 5] >> lane) & 1u);
      unsigned bal = __ballot_sync(0xffffffffu, on);
      if (on) list[n + __popc(bal & ((1u << lane) - 1u))] = static_cast<OutT>(base + lane);
      n += __popc(bal);
    }
    __syncwarp();
  } else {
    for (int t = lane; t < kend; t += 32) list[t] = static_cast<OutT>(t);
    n = kend;
  }
  __syncwarp();
  return n;
}

}  // namespace bsa
