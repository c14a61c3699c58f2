// Persistent, warp-specialised block-sparse FP8 attention prefill for sm_103a.
//
// One CTA per SM runs two independent pipelines.  Each pipeline claims (b, h, q-tile) tasks
// from a shared device counter (longest Q tile first) and owns 256 columns of tensor memory:
// S = Q K^T (fp32, 128 columns) and O (fp32, 128 columns).  Per pipeline:
//
//   producer warp   compacts the task's active KV tiles into a shared list (warp ballot),
//                   publishes the task, then streams Q and, tile by tile, the K pages, the
//                   per-token K descales and the V pages through TMA (2-stage rings; masked
//                   tiles are never addressed; a missing page is read at an out-of-range
//                   coordinate, which fills zeros).  The whole warp looks up the physical
//                   pages of 32 list tiles at once, a batch ahead of lane 0's copies.
//   MMA warp        one thread issues tcgen05.mma kind::f8f6f4: S(t+1) = Q K(t+1)^T as soon as
//                   the softmax has read S(t), then O (+)= P(t) V(t).
//   2 softmax       8 warps; warp (quarter q, sub-block u) owns rows 32q + 16u .. +15 of each
//   warpgroups      tile, and in it lane i takes row 32q + 16u + i%16 and column half i/16
//                   (tcgen05.ld.red shape 16x32bx2, which also returns the thread's maximum
//                   of the loaded values), so a row's two halves meet in one shuffle:
//                   scale, the row max, P = 2^(x - m) at the fixed P-scale (exact zeros past the
//                   causal edge and kv_len) rounded to e4m3 into a 128B-swizzled shared tile
//                   (the A operand of the PV MMA), O rescaled in TMEM when the row max moves,
//                   and the epilogue O * v_descale / l -> bf16, LSE -> fp32.
//
// Warps 0-3 are the producers and MMA issuers of the two pipelines; warps 4-19 are the four
// softmax warpgroups, which setmaxnreg gives most of the register file.
//
// Method: hpc-ops Block-Sparse FP8 Attention (活跃 tile 列表; 固定 P-scale 量化技巧) and the
// formula of Quant Block Sparse Attention (算子介绍).
#pragma once

#include "bsa_common.cuh"
#include "ptx_sm103.cuh"

namespace bsa {
namespace attn {

constexpr int NPIPE = 2;
constexpr int NTHREADS = 640;        // 4 control warps + 2 pipelines x 2 softmax warpgroups
constexpr int KSTAGES = 2;
constexpr int VSTAGES = 2;
constexpr int KDSTAGES = 2;
constexpr int MAX_SPLITS = 8;  // split-KV slices per task at most
constexpr int KD_STRIDE = TILE + 4;
__host__ __device__ constexpr int kd_index(int token) { return token + (token >= 64 ? 4 : 0); }
constexpr uint32_t TMEM_COLS = 512;  // per pipeline: S [0, 128), O [128, 256)
constexpr int CTRL_REGS = 56;
constexpr int SOFTMAX_REGS = 104;
// registers the split needs from the launch allocation (640 threads x 96 = 61440)
constexpr int SPLIT_REGS = 4 * 32 * CTRL_REGS + 16 * 32 * SOFTMAX_REGS;
static_assert(SPLIT_REGS <= NTHREADS * 96, "register split must fit 640 threads x 96 registers");

// The list is ascending and every row of a Q tile sees all keys below its first row's limit,
// so only the last two active tiles of a task can be partly hidden (causal edge, kv_len):
// the softmax needs just their indices, carried here.
struct TaskInfo {
  int b, h, qt;
  int n;          // tiles of this work item: list positions [lo, lo + n)
  int q0, q_len, kv_len;
  int tail0, tail1;  // the task's last two active tiles (the only ones with hidden keys)
  int lo, ntot;   // first list position of the item, length of the task's whole list
  int item, task;  // work-item index (task x split) and task index, for split-KV partials
  int split;       // this item's slice of the task (0 .. splits-1)
  int pad[2];
};

struct __align__(1024) Pipe {
  uint8_t q[TILE * HEAD_DIM];
  uint8_t k[KSTAGES][TILE * HEAD_DIM];
  uint8_t v[VSTAGES][TILE * HEAD_DIM];
  uint8_t p[TILE * HEAD_DIM];
  // per-token K descales of a tile; the second 64 tokens start 16 bytes late so that the two
  // column halves of a warp read different banks
  float kd[KDSTAGES][KD_STRIDE];
  TaskInfo info[2];
  uint32_t bitmap[KB_MAX / 32];
  int pg[2][32][4];  // physical pages of 32 consecutive list tiles, two batches (producer)
  uint64_t task_full[2], task_empty[2];
  uint64_t q_full, q_empty;
  uint64_t k_full[KSTAGES], k_empty[KSTAGES];
  uint64_t v_full[VSTAGES], v_empty[VSTAGES];
  uint64_t kd_full[KDSTAGES], kd_empty[KDSTAGES];
  uint64_t s_full, s_empty, p_full, o_done, o_empty, drain;
  int abort_flag;
};

struct __align__(1024) Smem {
  Pipe pipe[NPIPE];
  uint32_t tmem_base;
  // one task list of kb_pad(Kb) uint16 per pipeline follows the struct
};

__host__ __device__ constexpr int kb_pad(int Kb) { return (Kb + 7) & ~7; }

inline size_t smem_bytes(int Kb) {
  return sizeof(Smem) + NPIPE * (size_t)kb_pad(Kb) * sizeof(uint16_t) + 1024;
}
static_assert(sizeof(Smem) + NPIPE * kb_pad(KB_MAX) * sizeof(uint16_t) + 1024 <= 227 * 1024,
              "the longest task lists must fit one CTA's shared memory");

// Bounded mbarrier wait.  On timeout: report, raise the pipeline's abort flag and return false.
// Returns false without waiting once another role of the pipeline has aborted.
template <typename PipeT>
__device__ __forceinline__ bool wait_bar(const Params &p, PipeT &s, uint64_t *bar,
                                         uint32_t parity) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  // a probe suspends the thread for at most the launch's limit, so that a short limit holds
  const uint32_t hint = (uint32_t)min(p.wait_limit_ns, (unsigned long long)WAIT_LIMIT_NS);
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait_hint(bar, parity, hint)) return true;
    if ((it & 63u) == 1) {  // the first failed probe, then every 64th
      if (*(volatile int *)&s.abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > p.wait_limit_ns) {
        report(p, BSA_DEV_TIMEOUT);
        *(volatile int *)&s.abort_flag = 1;
        return false;
      }
    }
  }
}

// The softmax warps' waits after a first failed test, out of line so that their hot path
// carries only the test (the smaller loop body measurably helps the softmax).
template <typename PipeT>
__device__ __noinline__ bool wait_bar_warp_slow(const Params &p, PipeT &s, uint64_t *bar,
                                                uint32_t parity) {
  return __all_sync(0xffffffffu, wait_bar(p, s, bar, parity));
}

// Warp-uniform version for code followed by warp-collective instructions.
template <typename PipeT>
__device__ __forceinline__ bool wait_bar_warp(const Params &p, PipeT &s, uint64_t *bar,
                                              uint32_t parity) {
  if (__all_sync(0xffffffffu, ptx::mbar_try_wait(bar, parity))) return true;
  return wait_bar_warp_slow(p, s, bar, parity);
}

// Bounded wait that ignores the abort flag and the launch's wait limit (used to let in-flight
// async work land before the CTA exits).
__device__ __forceinline__ void drain_bar(uint64_t *bar, uint32_t parity) {
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > WAIT_LIMIT_NS) return;
  }
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

// Physical pages of the 128-token tile `tile` of sequence b (num_pages = read as zeros).
__device__ __forceinline__ int tile_pages(const Params &p, int b, int tile, int kv_len,
                                          int (&pgs)[4]) {
  const int npg = TILE / p.ps;
  int nvalid = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int pg = p.num_pages;
    if (i < npg && tile * TILE + i * p.ps < kv_len) {
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
  return nvalid;
}

// ===================================================================================== producer
__device__ __forceinline__ void run_producer(const Params &p, Pipe &s, uint16_t *list,
                                             const CUtensorMap *tmap_q,
                                             const CUtensorMap *tmap_k,
                                             const CUtensorMap *tmap_v) {
  const int lane = threadIdx.x & 31;
  const int per_qt = p.B * p.N1 * p.splits;  // work items per Q tile
  const int nitems = per_qt * p.Qb;
  const int npg = TILE / p.ps;
  int k = 0, qk = 0;
  uint32_t g = 0;
  bool ok = true;
  // Copies issued into each ring (lane 0): qk Q tiles; K, K-descale and V tiles for the g
  // finished tiles, or -- recorded only where a wait fails in the middle of a task -- fk >> 1 K
  // tiles (one descale tile fewer if fk & 1) and fv V tiles.
  uint32_t fk = ~0u, fv = 0;
  for (;;) {
    // claim the next work item: items are numbered by Q tile, descending, so the longest
    // causal tasks go first and a pipeline that finishes early takes the next one
    // (longest-first); with split-KV the slices of one task are consecutive items
    int o = 0;
    if (lane == 0) o = atomicAdd(p.task_counter, 1);
    o = __shfl_sync(0xffffffffu, o, 0);
    if (o >= nitems) break;
    const int qt = p.Qb - 1 - o / per_qt;
    const int rem = o % per_qt;
    const int split = rem % p.splits, bh = rem / p.splits;
    const int b = bh / p.N1, h = bh % p.N1;
    const TaskGeo geo = task_geometry(p, b, qt);
    if (!geo.valid) continue;
    const int slot = k & 1;
    if (k >= 2 &&
        !__all_sync(0xffffffffu, wait_bar(p, s, &s.task_empty[slot], ((k >> 1) - 1) & 1))) {
      ok = false;
      break;
    }
    // only this warp reads the list, and it has issued every load of the previous task
    __syncwarp();
    const int ntot = compact_task(p, b, h, qt, geo.kend, list, s.bitmap);
    // this item's slice of the task's list, by position (split-KV)
    const int lo = (int)((long long)split * ntot / p.splits);
    const int n = (int)((long long)(split + 1) * ntot / p.splits) - lo;
    if (lane == 0) {
      TaskInfo ti;
      ti.b = b;
      ti.h = h;
      ti.qt = qt;
      ti.n = n;
      ti.q0 = geo.q0;
      ti.q_len = geo.q_len;
      ti.kv_len = geo.kv_len;
      ti.tail0 = ntot >= 2 ? list[ntot - 2] : 0;
      ti.tail1 = ntot >= 1 ? list[ntot - 1] : 0;
      ti.lo = lo;
      ti.ntot = ntot;
      ti.item = o;
      ti.task = (b * p.N1 + h) * p.Qb + qt;
      ti.split = split;
      s.info[slot] = ti;
      ptx::mbar_arrive(&s.task_full[slot]);
    }
    ++k;
    if (n > 0) {
      const int g_kv = h / p.G;
      // The physical pages of list tiles lo + 32 j .. + 31 are looked up by the whole warp at
      // once (lane i: tile 32 j + i), one batch ahead of their use, so that the dependent
      // block_table loads do not sit between consecutive tiles' copies.
      int pf[4];
      auto lookup = [&](int t0) {
        const int t = t0 + lane;
        if (t < n) {
          tile_pages(p, b, list[lo + t], geo.kv_len, pf);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) pf[i] = p.num_pages;
        }
      };
      lookup(0);
      if (lane == 0) {
        if (qk >= 1 && !wait_bar(p, s, &s.q_empty, (qk - 1) & 1)) ok = false;
        if (ok) {
          ptx::mbar_arrive_expect_tx(&s.q_full, TILE * HEAD_DIM);
          const int tok0 = geo.q0 + qt * TILE;  // the Q box is 128 tokens of head h either way
          ptx::tma_load_3d(s.q, tmap_q, &s.q_full, 0, p.q_ntd ? tok0 : h, p.q_ntd ? h : tok0);
          ++qk;  // lane 0 counts the Q copies issued; the others take its count below
        }
      }
      int prev[4] = {0, 0, 0, 0};
      for (int t = 0; t <= n; ++t) {
        if ((t & 31) == 0 && t < n) {
          // batch t / 32 becomes current; start the next one
#pragma unroll
          for (int i = 0; i < 4; ++i) s.pg[(t >> 5) & 1][lane][i] = pf[i];
          __syncwarp();
          if (t + 32 < n) lookup(t + 32);
        }
        if (lane == 0 && ok) {
          int pgs[4] = {0, 0, 0, 0};
          if (t < n) {
#pragma unroll
            for (int i = 0; i < 4; ++i) pgs[i] = s.pg[(t >> 5) & 1][t & 31][i];
            const uint32_t gk = g + t;
            const int ks = gk % KSTAGES;
            if (gk >= KSTAGES && !wait_bar(p, s, &s.k_empty[ks], ((gk / KSTAGES) - 1) & 1)) {
              ok = false;  // K, descales and V issued for tiles < t, < t, < t - 1
              fk = gk << 1;
              fv = t >= 1 ? gk - 1 : g;
            } else {
              ptx::mbar_arrive_expect_tx(&s.k_full[ks], TILE * HEAD_DIM);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                if (i < npg)
                  ptx::tma_load_4d(s.k[ks] + i * p.ps * HEAD_DIM, tmap_k, &s.k_full[ks], 0,
                                   p.kv_nhd ? g_kv : 0, p.kv_nhd ? 0 : g_kv, pgs[i]);
              if (p.k_per_token) {
                const int ds = gk % KDSTAGES;
                if (gk >= KDSTAGES &&
                    !wait_bar(p, s, &s.kd_empty[ds], ((gk / KDSTAGES) - 1) & 1)) {
                  ok = false;  // K issued for tile t too, its descales not
                  fk = ((gk + 1) << 1) | 1u;
                  fv = t >= 1 ? gk - 1 : g;
                } else {
                  int nvalid = 0;
#pragma unroll
                  for (int i = 0; i < 4; ++i) nvalid += (i < npg && pgs[i] < p.num_pages);
                  ptx::mbar_arrive_expect_tx(&s.kd_full[ds], (uint32_t)(nvalid * p.ps * 4));
#pragma unroll
                  for (int i = 0; i < 4; ++i)
                    if (i < npg && pgs[i] < p.num_pages)
                      ptx::bulk_load(&s.kd[ds][kd_index(i * p.ps)],
                                     p.k_descale + ((size_t)pgs[i] * p.N2 + g_kv) * p.ps,
                                     (uint32_t)(p.ps * 4), &s.kd_full[ds]);
                }
              }
            }
          }
          if (ok && t >= 1) {
            // V of the previous tile: K runs one tile ahead of V, in the order the MMAs
            // consume them (S(t) is issued before PV(t-1))
            const uint32_t gv = g + t - 1;
            const int vs = gv % VSTAGES;
            if (gv >= VSTAGES && !wait_bar(p, s, &s.v_empty[vs], ((gv / VSTAGES) - 1) & 1)) {
              ok = false;  // K and descales issued for tiles <= t (the list has n), V for < t - 1
              fk = (g + min(t + 1, n)) << 1;
              fv = gv;
            } else {
              ptx::mbar_arrive_expect_tx(&s.v_full[vs], TILE * HEAD_DIM);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                if (i < npg)
                  ptx::tma_load_4d(s.v[vs] + i * p.ps * HEAD_DIM, tmap_v, &s.v_full[vs], 0,
                                   p.kv_nhd ? g_kv : 0, p.kv_nhd ? 0 : g_kv, prev[i]);
            }
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) prev[i] = pgs[i];
        }
        if ((t & 31) == 31 && !__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      }
      if (ok) g += n;  // lane 0's count is the one broadcast below
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    g = __shfl_sync(0xffffffffu, g, 0);
    qk = __shfl_sync(0xffffffffu, qk, 0);
    if (!ok) break;
  }
  // end-of-work marker
  if (ok) {
    const int slot = k & 1;
    if (k < 2 ||
        __all_sync(0xffffffffu, wait_bar(p, s, &s.task_empty[slot], ((k >> 1) - 1) & 1))) {
      if (lane == 0) {
        s.info[slot].n = -1;
        ptx::mbar_arrive(&s.task_full[slot]);
      }
    }
  }
  if (lane == 0 && *(volatile int *)&s.abort_flag) {
    // every copy issued must land before shared memory goes away: the last copy issued into
    // each slot of each ring completes its slot's latest phase, and a slot's phases complete
    // in order, so waiting for those phases covers every earlier copy too
    const bool mid = fk != ~0u;
    const uint32_t nk = mid ? fk >> 1 : g, nkd = nk - (mid ? (fk & 1u) : 0u), nv = mid ? fv : g;
    auto drain_ring = [&](uint64_t *full, uint32_t stages, uint32_t issued) {
      for (uint32_t x = issued >= stages ? issued - stages : 0; x < issued; ++x)
        drain_bar(&full[x % stages], (x / stages) & 1);
    };
    if (qk >= 1) drain_bar(&s.q_full, (qk - 1) & 1);
    drain_ring(s.k_full, KSTAGES, nk);
    drain_ring(s.v_full, VSTAGES, nv);
    if (p.k_per_token) drain_ring(s.kd_full, KDSTAGES, nkd);
  }
}

// ===================================================================================== MMA
__device__ __forceinline__ void run_mma(const Params &p, Pipe &s, uint32_t tmem) {
  constexpr uint32_t IDESC_S = ptx::idesc_e4m3_f32(128, 128, 0);   // B = K tile, K-major
  constexpr uint32_t IDESC_PV = ptx::idesc_e4m3_f32(128, 128, 1);  // B = V tile, MN-major
  const uint32_t tS = tmem, tO = tmem + 128;
  const uint32_t q_addr = ptx::smem_u32(s.q);
  const uint32_t p_addr = ptx::smem_u32(s.p);
  int k = 0, qk = 0;
  uint32_t g = 0;
  bool ok = true;
  auto issue_s = [&](uint32_t gs) -> bool {
    const int ks = gs % KSTAGES;
    if (!wait_bar(p, s, &s.k_full[ks], (gs / KSTAGES) & 1)) return false;
    if (gs >= 1 && !wait_bar(p, s, &s.s_empty, (gs - 1) & 1)) return false;
    ptx::tc_fence_after();
    const uint32_t k_addr = ptx::smem_u32(s.k[ks]);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      ptx::mma_f8_ss(tS, ptx::sdesc_sw128(q_addr + 32 * kk, 16, 1024),
                     ptx::sdesc_sw128(k_addr + 32 * kk, 16, 1024), IDESC_S, kk > 0);
    ptx::mma_commit(&s.k_empty[ks]);
    ptx::mma_commit(&s.s_full);
    return true;
  };
  for (; ok; ++k) {
    const int slot = k & 1;
    if (!wait_bar(p, s, &s.task_full[slot], (k >> 1) & 1)) {
      ok = false;
      break;
    }
    const int n = s.info[slot].n;
    if (n < 0) break;
    if (n > 0) {
      if (!wait_bar(p, s, &s.q_full, qk & 1)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      if (!issue_s(g)) {
        ok = false;
        break;
      }
      for (int t = 0; t < n; ++t) {
        const uint32_t gt = g + t;
        if (t + 1 < n) {
          if (!issue_s(gt + 1)) {
            ok = false;
            break;
          }
        } else {
          ptx::mma_commit(&s.q_empty);  // the task's last S has been issued
        }
        const int vs = gt % VSTAGES;
        if (!wait_bar(p, s, &s.p_full, gt & 1) ||
            !wait_bar(p, s, &s.v_full[vs], (gt / VSTAGES) & 1)) {
          ok = false;
          break;
        }
        // the previous task's epilogue must have read O before this task's first PV
        if (t == 0 && k >= 1 && !wait_bar(p, s, &s.o_empty, (k - 1) & 1)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t v_addr = ptx::smem_u32(s.v[vs]);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_f8_ss(tO, ptx::sdesc_sw128(p_addr + 32 * kk, 16, 1024),
                         ptx::sdesc_sw128(v_addr + 4096 * kk, 8192, 1024), IDESC_PV,
                         (t > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit(&s.v_empty[vs]);
        ptx::mma_commit(&s.o_done);
      }
      if (!ok) break;
      g += n;
      ++qk;
    } else if (k >= 1 && !wait_bar(p, s, &s.o_empty, (k - 1) & 1)) {
      ok = false;  // an empty task still takes its o_empty phase, keeping phases in order
      break;
    }
    ptx::mbar_arrive(&s.task_empty[slot]);
  }
  ptx::mma_commit(&s.drain);  // arrives once every MMA issued so far has finished
  drain_bar(&s.drain, 0);
}

// ===================================================================================== softmax
// Split-KV epilogue of one work item, thread (row r, column half): the item's O half-row
// (fp32, P-scale units, not normalised) and its (m, l) go to the workspace; the last of the
// task's items to finish the half-row merges the slices with log-sum-exp weights into the
// bf16 output, and the half-0 merger writes the LSE (the writes are fenced before the
// counter, the merger fences after it).  Out of line: it keeps the per-tile loop's register
// allocation independent of this path.
__device__ __noinline__ void split_epilogue(const Params &p, Pipe &s, const TaskInfo &ti,
                                            uint32_t tO, int r, int half, int col0, int n,
                                            float m, float l_row, float vd, bool row_ok,
                                            int tok, int h) {
  const size_t prow = (size_t)ti.item * TILE + r;
  float4 *po = reinterpret_cast<float4 *>(p.part_o + prow * HEAD_DIM + col0);
#pragma unroll 1
  for (int c = 0; c < 2; ++c) {
    uint32_t o[32];
    if (n > 0) {
      ptx::tmem_ld16x2_32<64>(tO + c * 32, o);
      ptx::tmem_ld_wait(o);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) o[j] = 0u;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      po[c * 8 + j] = make_float4(u2f(o[4 * j]), u2f(o[4 * j + 1]), u2f(o[4 * j + 2]),
                                  u2f(o[4 * j + 3]));
  }
  reinterpret_cast<float2 *>(p.part_ml)[prow * 2 + half] = make_float2(m, l_row);
  ptx::tc_fence_before();
  ptx::mbar_arrive(&s.o_empty);
  __threadfence();
  int *cnt = p.row_cnt + ((size_t)ti.task * TILE + r) * 2 + half;
  if (atomicAdd(cnt, 1) == p.splits - 1) {
    __threadfence();
    const size_t row0 = (size_t)(ti.item - ti.split) * TILE + r;  // slice 0 of the task
    const float2 *ml = reinterpret_cast<const float2 *>(p.part_ml);
    float w[MAX_SPLITS];
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < MAX_SPLITS; ++c) {
      w[c] = 0.f;
      if (c < p.splits) M = fmaxf(M, __ldcg(&ml[(row0 + (size_t)c * TILE) * 2 + half]).x);
    }
    float L = 0.f;
#pragma unroll
    for (int c = 0; c < MAX_SPLITS; ++c)
      if (c < p.splits) {
        const float2 v = __ldcg(&ml[(row0 + (size_t)c * TILE) * 2 + half]);
        if (v.x != -INFINITY && v.y > 0.f) {
          w[c] = ptx::ex2_approx(v.x - M);
          L += w[c] * v.y;
        }
      }
    const bool any = M != -INFINITY && L > 0.f;
    const float norm = any ? vd / L : 0.f;
    uint4 *orow =
        reinterpret_cast<uint4 *>(p.out + ((size_t)tok * p.N1 + h) * HEAD_DIM + col0);
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {  // 16 columns at a time
      float acc[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[j] = 0.f;
#pragma unroll
      for (int c = 0; c < MAX_SPLITS; ++c) {
        if (c >= p.splits) break;
        const float wc = w[c] * norm;
        const float4 *src = reinterpret_cast<const float4 *>(
            p.part_o + (row0 + (size_t)c * TILE) * HEAD_DIM + col0 + q * 16);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float4 v = __ldcg(src + j);
          acc[4 * j] += wc * v.x;
          acc[4 * j + 1] += wc * v.y;
          acc[4 * j + 2] += wc * v.z;
          acc[4 * j + 3] += wc * v.w;
        }
      }
      uint32_t wb[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        __nv_bfloat162 v2 = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
        wb[j] = *reinterpret_cast<uint32_t *>(&v2);
      }
      if (row_ok) {
        orow[q * 2] = make_uint4(wb[0], wb[1], wb[2], wb[3]);
        orow[q * 2 + 1] = make_uint4(wb[4], wb[5], wb[6], wb[7]);
      }
    }
    if (half == 0 && row_ok && p.lse)
      p.lse[(size_t)h * p.T + tok] =
          any ? (M + __log2f(L)) * 0.69314718055994531f - p.ln_pscale : -3.402823466e38f;
  }
}

// Thread (row r, half h) owns columns [64h, 64h + 64) of row r of every tile; `sub` selects
// which 16 rows of each 32-row TMEM quarter this warpgroup takes.
__device__ __forceinline__ void run_softmax(const Params &p, Pipe &s, uint32_t tmem, int sub) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;  // a warp may touch TMEM lanes 32*(warp%4) .. +31
  const int r = quad * 32 + sub * 16 + (lane & 15);
  const int half = lane >> 4;
  const int col0 = half * 64;
  const uint32_t tS = tmem + ((uint32_t)(quad * 32 + sub * 16) << 16);
  const uint32_t tO = tS + 128;
  uint8_t *prow = s.p + (r >> 3) * 1024 + (r & 7) * 128;
  int k = 0;
  uint32_t g = 0;
  for (;; ++k) {
    const int slot = k & 1;
    if (!wait_bar_warp(p, s, &s.task_full[slot], (k >> 1) & 1)) break;
    // the task's record stays put until this task's task_empty arrival: fields are read from
    // shared memory where they are used rather than held in registers across the tile loop
    const TaskInfo &ti = s.info[slot];
    const int n = ti.n;
    if (n < 0) break;
    // item tiles t >= t_hidden are the task's last two, the only ones with hidden keys
    const int t_hidden = ti.ntot - 2 - ti.lo;
    float row_scale;
    int causal_lim;  // keys j <= causal_lim are visible to row r
    {
      const int qt = ti.qt, h = ti.h, q_len = ti.q_len;
      const int tok = ti.q0 + qt * TILE + r;
      const float qd =
          r < min(TILE, q_len - qt * TILE)
              ? p.q_descale[(size_t)tok * p.qd_tok + (size_t)h * p.qd_head]
              : 0.f;
      row_scale = qd * p.scale_log2 * (p.k_per_token ? 1.f : p.k_descale[0]);
      causal_lim = qt * TILE + r + (ti.kv_len - q_len);
    }
    const bool neg_scale = row_scale < 0.f;
    const bool any_neg = __any_sync(0xffffffffu, neg_scale);
    // |scale| floored at 1e-30: a row whose descale is 0 then has logits of about 1e-23 in
    // place of exact zeros (the same P in fp32), and a hidden key's -inf stays -inf
    const float rs_abs = fmaxf(fabsf(row_scale), 1e-30f);
    const uint64_t rs2 = ptx::pk(rs_abs, rs_abs);
    float m = -INFINITY, l = 0.f;  // l: this half's share of the row sum (same m in both)
    // S is read with tcgen05.ld.red, which also returns the largest value the thread loaded.
    // With a per-tensor K descale and no negative row scale the logits are S times a positive
    // factor, so on tiles without hidden keys that maximum is the row-half maximum and the
    // max over the 64 values is skipped; a per-token K descale changes the order, so there
    // the maximum is taken after the multiply as before.
    const bool load_max = !p.k_per_token && !any_neg;
    bool ok = true;
    for (int t = 0; t < n; ++t) {
      const uint32_t gt = g + t;
      if (!wait_bar_warp(p, s, &s.s_full, gt & 1)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      uint32_t x[2][32];
      const bool red_tile = load_max && t < t_hidden;
      float mx_load;
      ptx::tmem_ld16x2_64_max<64>(tS, x[0], x[1], mx_load);
      ptx::tmem_ld_wait(x[0]);
      ptx::reg_fence(x[1]);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&s.s_empty);

      if (p.k_per_token) {
        const int ds = gt % KDSTAGES;
        if (!wait_bar_warp(p, s, &s.kd_full[ds], (gt / KDSTAGES) & 1)) {
          ok = false;
          break;
        }
        const ulonglong2 *kd4 = reinterpret_cast<const ulonglong2 *>(&s.kd[ds][kd_index(col0)]);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int j = 0; j < 32; j += 4) {
            const ulonglong2 kv = kd4[(c * 32 + j) >> 2];  // 4 descales per 16-byte load
            float a0, a1, a2, a3;
            ptx::upk(ptx::mul2(ptx::pk(u2f(x[c][j]), u2f(x[c][j + 1])), kv.x), a0, a1);
            ptx::upk(ptx::mul2(ptx::pk(u2f(x[c][j + 2]), u2f(x[c][j + 3])), kv.y), a2, a3);
            x[c][j] = f2u(a0);
            x[c][j + 1] = f2u(a1);
            x[c][j + 2] = f2u(a2);
            x[c][j + 3] = f2u(a3);
          }
        // the slot is released with the P hand-off below, after fence.proxy.async: these are
        // generic-proxy reads of memory the next bulk copy (async proxy) rewrites, and only a
        // proxy fence orders the two
      }
      // a negative scale (never produced by amax/448 descales, but legal) is folded into the
      // values so that one row-max path serves every row
      if (any_neg && neg_scale) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j) x[c][j] ^= 0x80000000u;
      }
      // hidden keys (past the causal edge or kv_len) take the logit -inf: they neither raise
      // the max nor add to P.  Only the task's last two tiles can hold any.
      if (t >= t_hidden) {
        const int tile = (t == t_hidden) ? ti.tail0 : ti.tail1;
        int lim = ti.kv_len - tile * TILE;  // visible keys of the tile
        if (p.causal) lim = min(lim, causal_lim - tile * TILE + 1);
        lim -= col0;                        // ... of this thread's half
        if (__any_sync(0xffffffffu, lim < 64)) {
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c * 32 + j >= lim) x[c][j] = f2u(-INFINITY);
        }
      }
      float mx = mx_load;
      if (!red_tile) {
        float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          a0 = ptx::max3(a0, u2f(x[0][j]), u2f(x[0][j + 1]));
          a1 = ptx::max3(a1, u2f(x[0][j + 2]), u2f(x[0][j + 3]));
          a2 = ptx::max3(a2, u2f(x[1][j]), u2f(x[1][j + 1]));
          a3 = ptx::max3(a3, u2f(x[1][j + 2]), u2f(x[1][j + 3]));
        }
        mx = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));  // the row's other half
      // largest scaled logit of the tile so far (log2 units); -inf while every key is hidden
      const float m_new = fmaxf(m, mx * rs_abs);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ptx::ex2_approx(m - m_use);
      const uint64_t b2 = ptx::pk(p.log2_pscale - m_use, p.log2_pscale - m_use);
      uint32_t packed[16];          // this half of the row of P as e4m3, 4 keys per word
      uint64_t acc0 = 0, acc1 = 0;  // packed partial sums (the 0.0f bit pattern is 0)
#pragma unroll
      for (int c = 0; c < 2; ++c)
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float e0, e1, e2, e3;
          ptx::upk(ptx::fma2(ptx::pk(u2f(x[c][j]), u2f(x[c][j + 1])), rs2, b2), e0, e1);
          ptx::upk(ptx::fma2(ptx::pk(u2f(x[c][j + 2]), u2f(x[c][j + 3])), rs2, b2), e2, e3);
          const float p0 = ptx::ex2_approx(e0), p1 = ptx::ex2_approx(e1);
          const float p2 = ptx::ex2_approx(e2), p3 = ptx::ex2_approx(e3);
          acc0 = ptx::add2(acc0, ptx::pk(p0, p1));
          acc1 = ptx::add2(acc1, ptx::pk(p2, p3));
          packed[(c * 32 + j) >> 2] = ptx::cvt_e4m3x4(p0, p1, p2, p3);
        }
      {
        float s0, s1, s2, s3;
        ptx::upk(acc0, s0, s1);
        ptx::upk(acc1, s2, s3);
        l = alpha * l + ((s0 + s1) + (s2 + s3));
        m = m_new;
      }
      if (t > 0) {
        // PV(t-1) done: the P tile may be overwritten and O is stable for the rescale
        if (!wait_bar_warp(p, s, &s.o_done, (gt - 1) & 1)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
      }
      // row r of the P tile: 8-row groups 1024 B apart, rows 128 B apart, the 16-byte chunk q
      // of a row at chunk position q ^ (r % 8) (128-byte swizzle); this half owns chunks
      // 4*half .. 4*half + 3
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4 *>(prow + (((4 * half + q) ^ (r & 7)) << 4)) =
            make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
      ptx::fence_proxy_async_smem();
      if (t > 0 && !__all_sync(0xffffffffu, alpha == 1.f)) {
        // O *= alpha on this thread's 64 columns
        const uint64_t a2 = ptx::pk(alpha, alpha);
        uint32_t o[2][32];
        ptx::tmem_ld16x2_64<64>(tO, o[0], o[1]);
        ptx::tmem_ld_wait(o[0]);
        ptx::reg_fence(o[1]);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            float a, b3;
            ptx::upk(ptx::mul2(ptx::pk(u2f(o[c][j]), u2f(o[c][j + 1])), a2), a, b3);
            o[c][j] = f2u(a);
            o[c][j + 1] = f2u(b3);
          }
          ptx::tmem_st16x2_32<64>(tO + c * 32, o[c]);
        }
        ptx::tmem_st_wait();
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&s.p_full);
      if (p.k_per_token) ptx::mbar_arrive(&s.kd_empty[gt % KDSTAGES]);
    }
    if (!ok) break;
    // ------------------------------------------------------------------------- epilogue
    const int h = ti.h, qt = ti.qt;
    const bool row_ok = r < min(TILE, ti.q_len - qt * TILE);
    const int tok = ti.q0 + qt * TILE + r;
    const int g_kv = h / p.G;
    const float l_row = l + __shfl_xor_sync(0xffffffffu, l, 16);  // both halves share m
    if (n > 0) {
      if (!wait_bar_warp(p, s, &s.o_done, (g + n - 1) & 1)) break;
      ptx::tc_fence_after();
    }
    // a row saw a visible key iff its running max is finite; l_row carries the P-scale
    const bool seen = m != -INFINITY && l_row > 0.f;
    const float vd = p.v_per_head ? p.v_descale[g_kv] : p.v_descale[0];
    const float osc = seen ? vd / l_row : 0.f;
    if (p.splits > 1) {
      split_epilogue(p, s, ti, tO, r, half, col0, n, m, l_row, vd, row_ok, tok, h);
    } else {
      const uint64_t osc2 = ptx::pk(osc, osc);
      // O goes out through this warp's 16 rows of the P tile (PV has finished reading them):
      // each 32-column round is staged row-wise and copied out so that a store instruction
      // writes whole 64-byte row segments instead of 16 bytes from each of 32 rows.  Staged
      // row i holds its two 64-byte segments as chunks 0-3 and 4-7, chunk c at position
      // c ^ (i % 8) so that both the staging and the copy-out touch every bank once per 128 B.
      const int r0 = quad * 32 + sub * 16;
      uint8_t *stage = s.p + r0 * 128;
      const int i = lane & 15;
      const int rows_valid = min(TILE, ti.q_len - qt * TILE);
      uint8_t *orow0 = reinterpret_cast<uint8_t *>(p.out) +
                       ((size_t)(ti.q0 + qt * TILE + r0) * p.N1 + h) * (HEAD_DIM * 2);
      const size_t row_bytes = (size_t)p.N1 * HEAD_DIM * 2;
  #pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        if (n > 0) {
          ptx::tmem_ld16x2_32<64>(tO + c * 32, o);
          ptx::tmem_ld_wait(o);
        } else {
  #pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = 0u;
        }
        uint32_t w[16];
  #pragma unroll
        for (int j = 0; j < 16; ++j) {
          float a, b3;
          ptx::upk(ptx::mul2(ptx::pk(u2f(o[2 * j]), u2f(o[2 * j + 1])), osc2), a, b3);
          __nv_bfloat162 v2 = __floats2bfloat162_rn(a, b3);
          w[j] = *reinterpret_cast<uint32_t *>(&v2);
        }
  #pragma unroll
        for (int q = 0; q < 4; ++q)
          *reinterpret_cast<uint4 *>(stage + i * 128 + (((4 * half + q) ^ (i & 7)) << 4)) =
              make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        __syncwarp();
  #pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int i2 = kk * 4 + (lane >> 3), c8 = lane & 7;
          const uint4 v = *reinterpret_cast<const uint4 *>(stage + i2 * 128 + ((c8 ^ (i2 & 7)) << 4));
          if (r0 + i2 < rows_valid)
            *reinterpret_cast<uint4 *>(orow0 + i2 * row_bytes + (c8 >> 2) * 128 + c * 64 +
                                       (c8 & 3) * 16) = v;
        }
        __syncwarp();
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&s.o_empty);
      if (half == 0 && row_ok && p.lse) {
        const float lse = seen ? (m + __log2f(l_row)) * 0.69314718055994531f - p.ln_pscale
                               : -3.402823466e38f;
        p.lse[(size_t)h * p.T + tok] = lse;
      }
    }
    ptx::mbar_arrive(&s.task_empty[slot]);
    g += n;
  }
}

__global__ void __launch_bounds__(NTHREADS, 1)
    bsa_attention_kernel(const __grid_constant__ Params p,
                         const __grid_constant__ CUtensorMap tmap_q,
                         const __grid_constant__ CUtensorMap tmap_k,
                         const __grid_constant__ CUtensorMap tmap_v) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment (128B-swizzled tiles) by pointer arithmetic on smem_raw, so that the
  // compiler still knows every access through `base` is a shared-memory access
  uint8_t *base = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  Smem &sm = *reinterpret_cast<Smem *>(base);
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x < NPIPE) {
    Pipe &s = sm.pipe[threadIdx.x];
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&s.task_full[i], 1);
      ptx::mbar_init(&s.task_empty[i], 256 + 1);  // both softmax warpgroups + the MMA thread
    }
    ptx::mbar_init(&s.q_full, 1);
    ptx::mbar_init(&s.q_empty, 1);
    for (int i = 0; i < KSTAGES; ++i) {
      ptx::mbar_init(&s.k_full[i], 1);
      ptx::mbar_init(&s.k_empty[i], 1);
    }
    for (int i = 0; i < VSTAGES; ++i) {
      ptx::mbar_init(&s.v_full[i], 1);
      ptx::mbar_init(&s.v_empty[i], 1);
    }
    for (int i = 0; i < KDSTAGES; ++i) {
      ptx::mbar_init(&s.kd_full[i], 1);
      ptx::mbar_init(&s.kd_empty[i], 256);
    }
    ptx::mbar_init(&s.s_full, 1);
    ptx::mbar_init(&s.s_empty, 256);
    ptx::mbar_init(&s.p_full, 256);
    ptx::mbar_init(&s.o_done, 1);
    ptx::mbar_init(&s.o_empty, 256);
    ptx::mbar_init(&s.drain, 1);
    s.abort_flag = 0;
    ptx::fence_mbarrier_init();
    if (threadIdx.x == 0) {
      ptx::prefetch_tmap(&tmap_q);
      ptx::prefetch_tmap(&tmap_k);
      ptx::prefetch_tmap(&tmap_v);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc(&sm.tmem_base, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();

  if (warp < 4) {
    ptx::regs_dec<CTRL_REGS>();
    const int pipe = warp >> 1;
    Pipe &s = sm.pipe[pipe];
    if ((warp & 1) == 0) {
      uint16_t *list = reinterpret_cast<uint16_t *>(base + sizeof(Smem)) + pipe * kb_pad(p.Kb);
      run_producer(p, s, list, &tmap_q, &tmap_k, &tmap_v);
    } else if ((threadIdx.x & 31) == 0) {
      run_mma(p, s, sm.tmem_base + 256u * pipe);
    }
  } else {
    ptx::regs_inc<SOFTMAX_REGS>();
    const int wg = (warp >> 2) - 1;  // 0..3: (pipeline, row sub-block)
    const int pipe = wg >> 1;
    run_softmax(p, sm.pipe[pipe], sm.tmem_base + 256u * pipe, wg & 1);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(sm.tmem_base, TMEM_COLS);
  }
}

}  // namespace attn
}  // namespace bsa
