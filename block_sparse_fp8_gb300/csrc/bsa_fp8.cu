// Block-sparse FP8 attention prefill over a paged KV cache, for GB300 (sm_103a).
//
// Two kernels:
//   * bsa_compact_kernel -- one warp per (b, h, qt) task writes the ascending list of active
//     KV tiles (warp ballot stream compaction; hpc-ops Block-Sparse FP8 Attention, section
//     活跃 tile 列表).  Exported for bit-exact checking; the attention kernel runs the same
//     device function on its own task.
//   * bsa_attention_kernel -- one CTA per (b, h, qt) task, warp-specialised:
//       warp 0     compacts the task's list into shared memory, then streams Q once and each
//                  active K/V tile through TMA, gathering 2 or 4 pages per 128-token tile via
//                  block_table (masked tiles are never addressed);
//       warp 1     allocates tensor memory and issues the tcgen05 MMAs (kind::f8f6f4):
//                  S = Q K^T into a double-buffered fp32 TMEM tile, O += P V into TMEM;
//       warps 2-5  one thread per query row: online softmax with -inf causal fill, P scaled
//                  by the fixed P-scale and rounded to e4m3 into shared memory (the A operand
//                  of the PV MMA), O rescaled in TMEM when the row max moves, and the
//                  epilogue O * v_descale / l -> bf16 and LSE -> fp32 (hpc-ops article,
//                  section 固定 P-scale 量化技巧; Quant Block Sparse Attention, 算子介绍).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "bsa_fp8.h"
#include "ptx_sm103.cuh"

namespace bsa {

constexpr int TILE = 128;
constexpr int HEAD_DIM = 128;
constexpr int KB_MAX = 4096;
constexpr int NSTAGE = 3;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s: far above any legitimate wait
constexpr int COMPACT_WARPS = 4;

struct Params {
  const uint8_t *q;
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
  int B, N1, N2, G, ps, max_q_len, max_kv_len, num_pages, L, T, Qb, Kb;
  int k_per_token, v_per_head, causal;
  float scale_log2;    // softmax_scale * log2(e)
  float log2_pscale;   // log2(p_scale)
  float ln_pscale;     // ln(p_scale)
};

__device__ __forceinline__ void report(const Params &p, int bits) {
  if (p.dev_status) atomicOr(p.dev_status, bits);
}

// Sequence geometry of task (b, qt).  kend = first KV tile that no row of the Q tile can see.
struct TaskGeo {
  int q0, q_len, kv_len, kend;
  bool valid;
};

__device__ TaskGeo task_geometry(const Params &p, int b, int qt) {
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

// Warp-cooperative active-tile compaction for task (b, h, qt): ascending, no repeats, < kend.
// `bitmap` is KB_MAX/32 words of this warp's shared memory (used by the index-list form).
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
    int len = p.sparse_seq_len[task];
    if (len < 0 || len > p.Kb) {
      if (lane == 0) report(p, BSA_DEV_BAD_INDEX);
      len = len < 0 ? 0 : p.Kb;
    }
    const int nwords = (kend + 31) >> 5;
    for (int w = lane; w < nwords; w += 32) bitmap[w] = 0u;
    __syncwarp();
    for (int e = lane; e < len; e += 32) {
      int t = p.sparse_indices[row + e];
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
// attention kernel
// ------------------------------------------------------------------------------------------

struct __align__(1024) Smem {
  uint8_t q[TILE * HEAD_DIM];               // Q tile, 128 rows x 128 B, 128B-swizzled
  uint8_t k[NSTAGE][TILE * HEAD_DIM];       // K tiles (ring)
  uint8_t v[NSTAGE][TILE * HEAD_DIM];       // V tiles (ring)
  uint8_t p[2][TILE * HEAD_DIM];            // e4m3 P tiles (double buffer), 128B-swizzled
  float kd[NSTAGE][TILE];                   // per-token K descales of the ring's tiles
  uint16_t list[KB_MAX];                    // active KV tiles of this task, ascending
  uint32_t bitmap[KB_MAX / 32];
  uint64_t q_full;
  uint64_t k_full[NSTAGE], v_full[NSTAGE], kv_empty[NSTAGE];
  uint64_t s_full[2], s_empty[2], p_full[2];
  uint64_t o_done, drain;
  uint32_t tmem_base;
  int n_active;
  int abort_flag;
  int q0, q_len, kv_len;
};

constexpr size_t SMEM_BYTES = sizeof(Smem) + 1024;

// Bounded mbarrier wait.  On timeout: report, raise the CTA's abort flag and return false.
// Also returns false (without waiting) once another role has aborted.
__device__ __forceinline__ bool wait_bar(const Params &p, Smem &s, uint64_t *bar,
                                         uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (*(volatile int *)&s.abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > WAIT_LIMIT_NS) {
        report(p, BSA_DEV_TIMEOUT);
        *(volatile int *)&s.abort_flag = 1;
        return false;
      }
    }
  }
}

// Bounded wait that ignores the abort flag (used to drain in-flight async work).
__device__ __forceinline__ void drain_bar(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > WAIT_LIMIT_NS) return;
  }
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

__global__ void __launch_bounds__(NUM_THREADS, 1)
    bsa_attention_kernel(const __grid_constant__ Params p,
                         const __grid_constant__ CUtensorMap tmap_q,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v) {
  extern __shared__ uint8_t smem_raw[];
  Smem &s = *reinterpret_cast<Smem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Task order: the Q-tile index runs slowest and descending, so the longest causal tasks
  // start first; heads of one KV group are neighbours (their K/V tiles meet in L2).
  const int per_qt = p.B * p.N1;
  const int qt = p.Qb - 1 - (int)(blockIdx.x / per_qt);
  const int rem = (int)(blockIdx.x % per_qt);
  const int b = rem / p.N1, h = rem % p.N1;
  const int g_kv = h / p.G;

  if (warp == 0) {
    TaskGeo g = task_geometry(p, b, qt);
    int n = g.valid ? compact_task(p, b, h, qt, g.kend, s.list, s.bitmap) : -1;
    if (lane == 0) {
      s.n_active = n;
      s.q0 = g.q0;
      s.q_len = g.q_len;
      s.kv_len = g.kv_len;
      s.abort_flag = 0;
    }
  }
  __syncthreads();
  const int n = s.n_active;
  if (n < 0) return;  // no rows of this sequence in this Q tile

  if (warp == 0 && lane == 0) {
    ptx::mbar_init(&s.q_full, 1);
    for (int i = 0; i < NSTAGE; ++i) {
      ptx::mbar_init(&s.k_full[i], 1);
      ptx::mbar_init(&s.v_full[i], 1);
      ptx::mbar_init(&s.kv_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&s.s_full[i], 1);
      ptx::mbar_init(&s.s_empty[i], 128);
      ptx::mbar_init(&s.p_full[i], 128);
    }
    ptx::mbar_init(&s.o_done, 1);
    ptx::mbar_init(&s.drain, 1);
    ptx::fence_mbarrier_init();
    ptx::prefetch_tmap(&tmap_q);
    ptx::prefetch_tmap(&tmap_k);
    ptx::prefetch_tmap(&tmap_v);
  } else if (warp == 1) {
    ptx::tmem_alloc(&s.tmem_base, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const int q0 = s.q0, q_len = s.q_len, kv_len = s.kv_len;
  const int off = kv_len - q_len;
  const int tok0 = q0 + qt * TILE;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (TMA)
    if (lane == 0 && n > 0) {
      ptx::mbar_arrive_expect_tx(&s.q_full, TILE * HEAD_DIM);
      ptx::tma_load_3d(s.q, &tmap_q, &s.q_full, 0, h, tok0);
      const int npg = TILE / p.ps;
      int issued = 0;
      for (int t = 0; t < n; ++t) {
        const int st = t % NSTAGE;
        if (t >= NSTAGE && !wait_bar(p, s, &s.kv_empty[st], ((t / NSTAGE) - 1) & 1)) break;
        const int tile = s.list[t];
        int pgs[4];
        int nvalid = 0;
        for (int i = 0; i < npg; ++i) {
          int pg = p.num_pages;  // out of range: TMA fills zeros
          if (tile * TILE + i * p.ps < kv_len) {
            const int lp = tile * npg + i;
            const int e = lp < p.L ? p.block_table[(size_t)b * p.L + lp] : -1;
            if (e < 0 || e >= p.num_pages)
              report(p, BSA_DEV_BAD_PAGE);
            else {
              pg = e;
              ++nvalid;
            }
          }
          pgs[i] = pg;
        }
        const uint32_t kd_bytes = p.k_per_token ? (uint32_t)(nvalid * p.ps * 4) : 0u;
        ptx::mbar_arrive_expect_tx(&s.k_full[st], TILE * HEAD_DIM + kd_bytes);
        for (int i = 0; i < npg; ++i) {
          ptx::tma_load_4d(s.k[st] + i * p.ps * HEAD_DIM, &tmap_k, &s.k_full[st], 0, 0, g_kv,
                           pgs[i]);
          if (p.k_per_token && pgs[i] < p.num_pages)
            ptx::bulk_load(&s.kd[st][i * p.ps],
                           p.k_descale + ((size_t)pgs[i] * p.N2 + g_kv) * p.ps,
                           (uint32_t)(p.ps * 4), &s.k_full[st]);
        }
        ptx::mbar_arrive_expect_tx(&s.v_full[st], TILE * HEAD_DIM);
        for (int i = 0; i < npg; ++i)
          ptx::tma_load_4d(s.v[st] + i * p.ps * HEAD_DIM, &tmap_v, &s.v_full[st], 0, 0, g_kv,
                           pgs[i]);
        issued = t + 1;
      }
      if (*(volatile int *)&s.abort_flag) {
        // let every copy still in flight land before the CTA's shared memory goes away
        drain_bar(&s.q_full, 0);
        for (int t = max(0, issued - NSTAGE); t < issued; ++t) {
          drain_bar(&s.k_full[t % NSTAGE], (t / NSTAGE) & 1);
          drain_bar(&s.v_full[t % NSTAGE], (t / NSTAGE) & 1);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (tcgen05)
    if (lane == 0 && n > 0) {
      constexpr uint32_t IDESC_S = ptx::idesc_e4m3_f32(128, 128, 0);   // B = K, K-major
      constexpr uint32_t IDESC_PV = ptx::idesc_e4m3_f32(128, 128, 1);  // B = V, MN-major
      const uint32_t tO = tmem + 256;
      const uint32_t q_addr = ptx::smem_u32(s.q);
      bool ok = wait_bar(p, s, &s.q_full, 0);
      ptx::tc_fence_after();
      auto issue_s = [&](int t) -> bool {
        const int st = t % NSTAGE;
        if (!wait_bar(p, s, &s.k_full[st], (t / NSTAGE) & 1)) return false;
        ptx::tc_fence_after();
        const uint32_t k_addr = ptx::smem_u32(s.k[st]);
        const uint32_t tS = tmem + (uint32_t)((t & 1) * 128);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_f8_ss(tS, ptx::sdesc_sw128(q_addr + 32 * kk, 16, 1024),
                         ptx::sdesc_sw128(k_addr + 32 * kk, 16, 1024), IDESC_S, kk > 0);
        ptx::mma_commit(&s.s_full[t & 1]);
        return true;
      };
      if (ok) ok = issue_s(0);
      if (ok && n > 1) ok = issue_s(1);
      for (int t = 0; ok && t < n; ++t) {
        const int st = t % NSTAGE;
        if (!wait_bar(p, s, &s.p_full[t & 1], (t >> 1) & 1)) break;
        if (!wait_bar(p, s, &s.v_full[st], (t / NSTAGE) & 1)) break;
        ptx::tc_fence_after();
        const uint32_t p_addr = ptx::smem_u32(s.p[t & 1]);
        const uint32_t v_addr = ptx::smem_u32(s.v[st]);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_f8_ss(tO, ptx::sdesc_sw128(p_addr + 32 * kk, 16, 1024),
                         ptx::sdesc_sw128(v_addr + 4096 * kk, 8192, 1024), IDESC_PV,
                         (t > 0 || kk > 0) ? 1u : 0u);
        if (t + NSTAGE < n) ptx::mma_commit(&s.kv_empty[st]);  // stage reloaded later
        ptx::mma_commit(&s.o_done);
        if (t + 2 < n) {
          if (!wait_bar(p, s, &s.s_empty[t & 1], (t >> 1) & 1)) break;
          if (!issue_s(t + 2)) break;
        }
      }
      if (*(volatile int *)&s.abort_flag) {
        ptx::mma_commit(&s.drain);  // arrives once every MMA issued so far has finished
        drain_bar(&s.drain, 0);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int quad = warp & 3;  // a warp may touch TMEM lanes 32*(warp%4) .. +31
    const int r = quad * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t tO = lane_base + 256;
    const int rows_valid = min(TILE, q_len - qt * TILE);
    const bool row_ok = r < rows_valid;
    const int tok = tok0 + r;
    const float qd = row_ok ? p.q_descale[(size_t)tok * p.N1 + h] : 0.f;
    const float row_scale = qd * p.scale_log2 * (p.k_per_token ? 1.f : p.k_descale[0]);
    const int causal_lim = qt * TILE + r + off;  // keys j <= causal_lim are visible
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int t = 0; t < n; ++t) {
      const int buf = t & 1, st = t % NSTAGE;
      const int tile = s.list[t];
      // wait outcomes are made warp-uniform: the tcgen05.ld/st below are warp-collective
      if (!__all_sync(0xffffffffu, wait_bar(p, s, &s.s_full[buf], (t >> 1) & 1))) {
        ok = false;
        break;
      }
      if (p.k_per_token &&
          !__all_sync(0xffffffffu, wait_bar(p, s, &s.k_full[st], (t / NSTAGE) & 1))) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      uint32_t x[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) ptx::tmem_ld32(lane_base + buf * 128 + c * 32, x[c]);
      ptx::tmem_ld_wait(x[0]);
      ptx::reg_fence(x[1]);
      ptx::reg_fence(x[2]);
      ptx::reg_fence(x[3]);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&s.s_empty[buf]);

      int lim = kv_len - tile * TILE;
      if (p.causal) lim = min(lim, causal_lim - tile * TILE + 1);
      float mx = -INFINITY;
      if (p.k_per_token) {
        const float4 *kd4 = reinterpret_cast<const float4 *>(s.kd[st]);
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const float4 kd = kd4[(c * 32 + j) >> 2];
            x[c][j + 0] = f2u(u2f(x[c][j + 0]) * row_scale * kd.x);
            x[c][j + 1] = f2u(u2f(x[c][j + 1]) * row_scale * kd.y);
            x[c][j + 2] = f2u(u2f(x[c][j + 2]) * row_scale * kd.z);
            x[c][j + 3] = f2u(u2f(x[c][j + 3]) * row_scale * kd.w);
          }
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j) x[c][j] = f2u(u2f(x[c][j]) * row_scale);
      }
      if (lim < TILE) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c * 32 + j >= lim) x[c][j] = f2u(-INFINITY);
      }
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int j = 0; j < 32; ++j) mx = fmaxf(mx, u2f(x[c][j]));
      const float m_new = fmaxf(m, mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ptx::ex2_approx(m - m_use);
      const float bias = p.log2_pscale - m_use;
      float sum = 0.f;
      uint32_t packed[32];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const float p0 = ptx::ex2_approx(u2f(x[c][j + 0]) + bias);
          const float p1 = ptx::ex2_approx(u2f(x[c][j + 1]) + bias);
          const float p2 = ptx::ex2_approx(u2f(x[c][j + 2]) + bias);
          const float p3 = ptx::ex2_approx(u2f(x[c][j + 3]) + bias);
          sum += (p0 + p1) + (p2 + p3);
          packed[(c * 32 + j) >> 2] =
              (uint32_t)ptx::cvt_e4m3x2(p0, p1) | ((uint32_t)ptx::cvt_e4m3x2(p2, p3) << 16);
        }
      // row r of the P tile: 8-row groups are 1024 B apart, rows 128 B apart, and the 16-byte
      // chunk c of a row sits at chunk position c ^ (r % 8) (128-byte swizzle)
      uint8_t *prow = s.p[buf] + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4 *>(prow + ((c ^ (r & 7)) << 4)) =
            make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
      l = alpha * l + sum;
      m = m_new;
      ptx::fence_proxy_async_smem();
      if (t > 0) {
        if (!__all_sync(0xffffffffu, wait_bar(p, s, &s.o_done, (t - 1) & 1))) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        if (!__all_sync(0xffffffffu, alpha == 1.f)) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            ptx::tmem_ld32(tO + c * 32, o);
            ptx::tmem_ld_wait(o);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = f2u(u2f(o[j]) * alpha);
            ptx::tmem_st32(tO + c * 32, o);
          }
          ptx::tmem_st_wait();
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&s.p_full[buf]);
    }

    if (ok && n > 0 && !__all_sync(0xffffffffu, wait_bar(p, s, &s.o_done, (n - 1) & 1)))
      ok = false;
    if (ok) {
      ptx::tc_fence_after();
      const float vd = p.v_per_head ? p.v_descale[g_kv] : p.v_descale[0];
      const float oscale = l > 0.f ? vd / l : 0.f;  // l already carries the P-scale
      uint4 *orow = reinterpret_cast<uint4 *>(p.out + ((size_t)tok * p.N1 + h) * HEAD_DIM);
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        if (n > 0) {
          ptx::tmem_ld32(tO + c * 32, o);
          ptx::tmem_ld_wait(o);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          __nv_bfloat162 v2 =
              __floats2bfloat162_rn(u2f(o[2 * j]) * oscale, u2f(o[2 * j + 1]) * oscale);
          w[j] = *reinterpret_cast<uint32_t *>(&v2);
        }
        if (row_ok) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            orow[c * 4 + j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        }
      }
      if (row_ok && p.lse) {
        const float lse = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f - p.ln_pscale
                                  : -3.402823466e38f;
        p.lse[(size_t)h * p.T + tok] = lse;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
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
  if (cdiv(d->max_kv_len, TILE) > KB_MAX) return BSA_ERR_UNSUPPORTED;
  if ((long long)d->B * d->N1 * cdiv(d->max_q_len, TILE) > 0x7fffffffLL)
    return BSA_ERR_UNSUPPORTED;
  return BSA_OK;
}

static bsa_status_t check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return BSA_ERR_CUDA;
  static int checked[64] = {0};  // 0 unknown, 1 ok, 2 unsupported
  if (dev < 0 || dev >= 64) return BSA_ERR_UNSUPPORTED;
  if (checked[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return BSA_ERR_CUDA;
    bool ok = major == 10 && minor == 3;
    if (ok && cudaFuncSetAttribute(bsa_attention_kernel,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)SMEM_BYTES) != cudaSuccess)
      return BSA_ERR_CUDA;
    checked[dev] = ok ? 1 : 2;
  }
  return checked[dev] == 1 ? BSA_OK : BSA_ERR_UNSUPPORTED;
}

static Params make_params(const bsa_fp8_dims_t *d) {
  Params p;
  memset(&p, 0, sizeof(p));
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

extern "C" size_t bsa_fp8_prefill_workspace_size(const bsa_fp8_dims_t *dims) {
  (void)dims;
  return 0;  // lists live in each CTA's shared memory
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
  st = check_device();
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
  (void)workspace;
  (void)workspace_bytes;
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
      (p.k_per_token && !aligned16(k_descale)) || !aligned16(out_bf16))
    return BSA_ERR_INVALID_ARGUMENT;
  st = check_device();
  if (st != BSA_OK) return st;

  p.q = static_cast<const uint8_t *>(q);
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
  p.scale_log2 = (float)((double)softmax_scale * 1.4426950408889634);
  p.log2_pscale = (float)std::log2((double)p_scale);
  p.ln_pscale = (float)std::log((double)p_scale);

  CUtensorMap tq, tk, tv;
  {
    cuuint64_t gd[3] = {HEAD_DIM, (cuuint64_t)p.N1, (cuuint64_t)p.T};
    cuuint64_t gs[2] = {HEAD_DIM, (cuuint64_t)p.N1 * HEAD_DIM};
    cuuint32_t box[3] = {HEAD_DIM, 1, TILE};
    if (!encode_map(&tq, q, 3, gd, gs, box)) return BSA_ERR_CUDA;
  }
  {
    cuuint64_t gd[4] = {HEAD_DIM, (cuuint64_t)p.ps, (cuuint64_t)p.N2, (cuuint64_t)p.num_pages};
    cuuint64_t gs[3] = {HEAD_DIM, (cuuint64_t)p.ps * HEAD_DIM,
                        (cuuint64_t)p.N2 * p.ps * HEAD_DIM};
    cuuint32_t box[4] = {HEAD_DIM, (cuuint32_t)p.ps, 1, 1};
    if (!encode_map(&tk, k_pages, 4, gd, gs, box)) return BSA_ERR_CUDA;
    if (!encode_map(&tv, v_pages, 4, gd, gs, box)) return BSA_ERR_CUDA;
  }
  bsa_attention_kernel<<<(unsigned)ntasks, NUM_THREADS, SMEM_BYTES, (cudaStream_t)stream>>>(
      p, tq, tk, tv);
  return cudaGetLastError() == cudaSuccess ? BSA_OK : BSA_ERR_CUDA;
}
