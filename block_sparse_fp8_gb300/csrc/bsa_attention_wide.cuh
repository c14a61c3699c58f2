// The prefill with 256-wide macro blocks: each online-softmax step takes two consecutive tiles
// of the active list (the Quant Block Sparse Attention kernel description pairs two sparse
// 128-token KV blocks into one 256-wide macro block; an odd last tile is a step of its own),
// so the row maximum, P's quantisation scale and the rescale of O move once per pair.
//
// One pipeline per CTA (one CTA per SM).  Tensor memory: S of the pair in columns [0, 256)
// (one N = 256 tcgen05.mma per K step over the two K tiles, which sit in adjacent shared
// slots), O in [256, 384).
//
//   warp 0          producer: compaction, Q, and per step the K tiles, their per-token
//                   descales and (one step behind) the V tiles of the pair, through TMA into
//                   2-step rings; pages looked up 32 tiles at a time by the whole warp.
//   warp 1          MMA issuer (one thread): S(s+1) once the softmax has read S(s), then
//                   O (+)= P0 V0 (+ P1 V1).
//   warps 4-19      softmax: warp w has quarter q = w % 4 of the rows, 16-row block u and tile
//                   h of the pair ((w / 4 - 1) = u + 2 h); a thread owns one half (64 columns)
//                   of one row of its tile (tcgen05.ld 16x32bx2).  The two warps of a row block
//                   exchange their row maxima through shared memory every step, guarded by an
//                   mbarrier (bounded wait), quantise P against the pair's maximum and each
//                   rescale their half of O's columns.
//
// Method: hpc-ops Block-Sparse FP8 Attention (活跃 tile 列表; 固定 P-scale 量化技巧) and
// Quant Block Sparse Attention (算子介绍; the kernel's 256-wide macro block).
#pragma once

#include "bsa_attention.cuh"

namespace bsa {
namespace attn_wide {

using attn::TaskInfo;
using attn::KD_STRIDE;
using attn::kd_index;
using attn::u2f;
using attn::f2u;

constexpr int NTHREADS = 640;  // warps 0-3 control (2, 3 idle), 4-19 softmax
constexpr int RING = 2;        // steps (tile pairs) in flight per ring
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t S_COL = 0, O_COL = 256;
constexpr int NSOFT = 512;     // softmax threads
constexpr int CTRL_REGS = attn::CTRL_REGS;
constexpr int SOFTMAX_REGS = attn::SOFTMAX_REGS;
constexpr int SPLIT_REGS = attn::SPLIT_REGS;

struct __align__(1024) Pipe {
  uint8_t q[TILE * HEAD_DIM];
  uint8_t k[RING][2][TILE * HEAD_DIM];  // a step's two K tiles are adjacent (one N=256 operand)
  uint8_t v[RING][2][TILE * HEAD_DIM];
  uint8_t p[2][TILE * HEAD_DIM];        // P of the pair's two tiles
  float kd[RING][2][KD_STRIDE];
  float xmax[2][2][TILE];  // row maxima of the two tiles, by step parity
  float xsum[2][TILE];     // row sums of the two tiles (epilogue)
  TaskInfo info[2];
  uint32_t bitmap[KB_MAX / 32];
  int pg[2][32][4];
  uint64_t task_full[2], task_empty[2];
  uint64_t q_full, q_empty;
  uint64_t k_full[RING], k_empty[RING];
  uint64_t v_full[RING], v_empty[RING];
  uint64_t kd_full[RING], kd_empty[RING];
  uint64_t s_full, s_empty, p_full, o_done, o_empty, drain;
  uint64_t xch[8];  // per (quarter, row block): both tile warps published their maxima
  int abort_flag;
};

struct __align__(1024) Smem {
  Pipe pipe;
  uint32_t tmem_base;
};

inline size_t smem_bytes(int Kb) {
  return sizeof(Smem) + (size_t)attn::kb_pad(Kb) * sizeof(uint16_t) + 1024;
}
static_assert(sizeof(Smem) + attn::kb_pad(KB_MAX) * sizeof(uint16_t) + 1024 <= 227 * 1024,
              "the longest task list must fit one CTA's shared memory");

__device__ __forceinline__ int steps_of(int n) { return (n + 1) >> 1; }
// tiles of step j of an item with n tiles: two, or one for an odd last step
__device__ __forceinline__ int tiles_in_step(int n, int j) { return 2 * j + 1 < n ? 2 : 1; }

// ===================================================================================== producer
__device__ __forceinline__ void run_producer(const Params &p, Pipe &s, uint16_t *list,
                                             const CUtensorMap *tmap_q,
                                             const CUtensorMap *tmap_k,
                                             const CUtensorMap *tmap_v) {
  const int lane = threadIdx.x & 31;
  const int per_qt = p.B * p.N1;  // work items per Q tile (no split-KV here)
  const int nitems = per_qt * p.Qb;
  const int npg = TILE / p.ps;
  int k = 0, qk = 0;
  uint32_t g = 0;  // steps of the finished tasks
  bool ok = true;
  // copies issued (lane 0): qk Q tiles; K, descale and V steps of the g finished steps, or --
  // recorded only where a wait fails inside a task -- fk >> 1 K steps (one descale step
  // fewer if fk & 1) and fv V steps
  uint32_t fk = ~0u, fv = 0;
  for (;;) {
    int o = 0;
    if (lane == 0) o = atomicAdd(p.task_counter, 1);
    o = __shfl_sync(0xffffffffu, o, 0);
    if (o >= nitems) break;
    const int qt = p.Qb - 1 - o / per_qt;
    const int bh = o % per_qt;
    const int b = bh / p.N1, h = bh % p.N1;
    const TaskGeo geo = task_geometry(p, b, qt);
    if (!geo.valid) continue;
    const int slot = k & 1;
    if (k >= 2 &&
        !__all_sync(0xffffffffu, attn::wait_bar(p, s, &s.task_empty[slot], ((k >> 1) - 1) & 1))) {
      ok = false;
      break;
    }
    __syncwarp();
    const int n = compact_task(p, b, h, qt, geo.kend, list, s.bitmap);
    if (lane == 0) {
      TaskInfo ti;
      ti.b = b;
      ti.h = h;
      ti.qt = qt;
      ti.n = n;
      ti.q0 = geo.q0;
      ti.q_len = geo.q_len;
      ti.kv_len = geo.kv_len;
      ti.tail0 = n >= 2 ? list[n - 2] : 0;
      ti.tail1 = n >= 1 ? list[n - 1] : 0;
      ti.lo = 0;
      ti.ntot = n;
      ti.item = o;
      ti.task = (b * p.N1 + h) * p.Qb + qt;
      ti.split = 0;
      s.info[slot] = ti;
      ptx::mbar_arrive(&s.task_full[slot]);
    }
    ++k;
    if (n > 0) {
      const int g_kv = h / p.G;
      const int nsteps = steps_of(n);
      int pf[4];
      auto lookup = [&](int t0) {
        const int t = t0 + lane;
        if (t < n) {
          attn::tile_pages(p, b, list[t], geo.kv_len, pf);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) pf[i] = p.num_pages;
        }
      };
      lookup(0);
      if (lane == 0) {
        if (qk >= 1 && !attn::wait_bar(p, s, &s.q_empty, (qk - 1) & 1)) ok = false;
        if (ok) {
          ptx::mbar_arrive_expect_tx(&s.q_full, TILE * HEAD_DIM);
          const int tok0 = geo.q0 + qt * TILE;
          ptx::tma_load_3d(s.q, tmap_q, &s.q_full, 0, p.q_ntd ? tok0 : h, p.q_ntd ? h : tok0);
          ++qk;
        }
      }
      // K and descales of step j, V of step j - 1; tile t's pages in s.pg[(t / 32) % 2][t % 32]
      for (int j = 0; j <= nsteps; ++j) {
        const int t0 = 2 * j;
        if ((t0 & 31) == 0 && t0 < n) {
#pragma unroll
          for (int i = 0; i < 4; ++i) s.pg[(t0 >> 5) & 1][lane][i] = pf[i];
          __syncwarp();
          if (t0 + 32 < n) lookup(t0 + 32);
        }
        if (lane == 0 && ok) {
          if (j < nsteps) {
            const int nt = tiles_in_step(n, j);
            const uint32_t gk = g + j;
            const int ks = gk % RING;
            if (gk >= RING && !attn::wait_bar(p, s, &s.k_empty[ks], ((gk / RING) - 1) & 1)) {
              ok = false;  // K, descales issued for steps < j, V for < j - 1
              fk = gk << 1;
              fv = j >= 1 ? gk - 1 : g;
            } else {
              ptx::mbar_arrive_expect_tx(&s.k_full[ks], (uint32_t)(nt * TILE * HEAD_DIM));
              for (int u = 0; u < nt; ++u) {
                const int t = t0 + u;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  if (i < npg)
                    ptx::tma_load_4d(s.k[ks][u] + i * p.ps * HEAD_DIM, tmap_k, &s.k_full[ks],
                                     0, p.kv_nhd ? g_kv : 0, p.kv_nhd ? 0 : g_kv,
                                     s.pg[(t >> 5) & 1][t & 31][i]);
              }
              if (p.k_per_token) {
                if (gk >= RING &&
                    !attn::wait_bar(p, s, &s.kd_empty[ks], ((gk / RING) - 1) & 1)) {
                  ok = false;  // K issued for step j too, its descales not
                  fk = ((gk + 1) << 1) | 1u;
                  fv = j >= 1 ? gk - 1 : g;
                } else {
                  int nvalid = 0;
                  for (int u = 0; u < nt; ++u)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                      nvalid += (i < npg && s.pg[((t0 + u) >> 5) & 1][(t0 + u) & 31][i] <
                                                p.num_pages);
                  ptx::mbar_arrive_expect_tx(&s.kd_full[ks], (uint32_t)(nvalid * p.ps * 4));
                  for (int u = 0; u < nt; ++u) {
                    const int t = t0 + u;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                      const int pg = s.pg[(t >> 5) & 1][t & 31][i];
                      if (i < npg && pg < p.num_pages)
                        ptx::bulk_load(&s.kd[ks][u][kd_index(i * p.ps)],
                                       p.k_descale + ((size_t)pg * p.N2 + g_kv) * p.ps,
                                       (uint32_t)(p.ps * 4), &s.kd_full[ks]);
                    }
                  }
                }
              }
            }
          }
          if (ok && j >= 1) {
            const int jv = j - 1, ntv = tiles_in_step(n, jv);
            const uint32_t gv = g + jv;
            const int vs = gv % RING;
            if (gv >= RING && !attn::wait_bar(p, s, &s.v_empty[vs], ((gv / RING) - 1) & 1)) {
              ok = false;  // K and descales issued for steps <= j (the item has nsteps)
              fk = (g + min(j + 1, nsteps)) << 1;
              fv = gv;
            } else {
              ptx::mbar_arrive_expect_tx(&s.v_full[vs], (uint32_t)(ntv * TILE * HEAD_DIM));
              for (int u = 0; u < ntv; ++u) {
                const int t = 2 * jv + u;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  if (i < npg)
                    ptx::tma_load_4d(s.v[vs][u] + i * p.ps * HEAD_DIM, tmap_v, &s.v_full[vs],
                                     0, p.kv_nhd ? g_kv : 0, p.kv_nhd ? 0 : g_kv,
                                     s.pg[(t >> 5) & 1][t & 31][i]);
              }
            }
          }
        }
        if ((j & 15) == 15 && !__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) break;
      }
      if (ok) g += nsteps;
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    g = __shfl_sync(0xffffffffu, g, 0);
    qk = __shfl_sync(0xffffffffu, qk, 0);
    if (!ok) break;
  }
  if (ok) {
    const int slot = k & 1;
    if (k < 2 ||
        __all_sync(0xffffffffu, attn::wait_bar(p, s, &s.task_empty[slot], ((k >> 1) - 1) & 1))) {
      if (lane == 0) {
        s.info[slot].n = -1;
        ptx::mbar_arrive(&s.task_full[slot]);
      }
    }
  }
  if (lane == 0 && *(volatile int *)&s.abort_flag) {
    // every copy issued lands before shared memory goes away (see the 128-wide kernel)
    const bool mid = fk != ~0u;
    const uint32_t nk = mid ? fk >> 1 : g, nkd = nk - (mid ? (fk & 1u) : 0u), nv = mid ? fv : g;
    auto drain_ring = [&](uint64_t *full, uint32_t issued) {
      for (uint32_t x = issued >= RING ? issued - RING : 0; x < issued; ++x)
        attn::drain_bar(&full[x % RING], (x / RING) & 1);
    };
    if (qk >= 1) attn::drain_bar(&s.q_full, (qk - 1) & 1);
    drain_ring(s.k_full, nk);
    drain_ring(s.v_full, nv);
    if (p.k_per_token) drain_ring(s.kd_full, nkd);
  }
}

// ===================================================================================== MMA
__device__ __forceinline__ void run_mma(const Params &p, Pipe &s, uint32_t tmem) {
  constexpr uint32_t IDESC_S2 = ptx::idesc_e4m3_f32(128, 256, 0);  // B = the two K tiles
  constexpr uint32_t IDESC_S1 = ptx::idesc_e4m3_f32(128, 128, 0);  // B = one K tile
  constexpr uint32_t IDESC_PV = ptx::idesc_e4m3_f32(128, 128, 1);  // B = a V tile, MN-major
  const uint32_t tS = tmem + S_COL, tO = tmem + O_COL;
  const uint32_t q_addr = ptx::smem_u32(s.q);
  int k = 0, qk = 0;
  uint32_t g = 0;
  bool ok = true;
  auto issue_s = [&](uint32_t gs, int nt) -> bool {
    const int ks = gs % RING;
    if (!attn::wait_bar(p, s, &s.k_full[ks], (gs / RING) & 1)) return false;
    if (gs >= 1 && !attn::wait_bar(p, s, &s.s_empty, (gs - 1) & 1)) return false;
    ptx::tc_fence_after();
    const uint32_t k_addr = ptx::smem_u32(s.k[ks][0]);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
      ptx::mma_f8_ss(tS, ptx::sdesc_sw128(q_addr + 32 * kk, 16, 1024),
                     ptx::sdesc_sw128(k_addr + 32 * kk, 16, 1024), nt == 2 ? IDESC_S2 : IDESC_S1,
                     kk > 0);
    ptx::mma_commit(&s.k_empty[ks]);
    ptx::mma_commit(&s.s_full);
    return true;
  };
  for (; ok; ++k) {
    const int slot = k & 1;
    if (!attn::wait_bar(p, s, &s.task_full[slot], (k >> 1) & 1)) {
      ok = false;
      break;
    }
    const int n = s.info[slot].n;
    if (n < 0) break;
    if (n > 0) {
      const int nsteps = steps_of(n);
      if (!attn::wait_bar(p, s, &s.q_full, qk & 1)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      if (!issue_s(g, tiles_in_step(n, 0))) {
        ok = false;
        break;
      }
      for (int j = 0; j < nsteps; ++j) {
        const uint32_t gj = g + j;
        if (j + 1 < nsteps) {
          if (!issue_s(gj + 1, tiles_in_step(n, j + 1))) {
            ok = false;
            break;
          }
        } else {
          ptx::mma_commit(&s.q_empty);  // the task's last S has been issued
        }
        const int vs = gj % RING;
        if (!attn::wait_bar(p, s, &s.p_full, gj & 1) ||
            !attn::wait_bar(p, s, &s.v_full[vs], (gj / RING) & 1)) {
          ok = false;
          break;
        }
        if (j == 0 && k >= 1 && !attn::wait_bar(p, s, &s.o_empty, (k - 1) & 1)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const int nt = tiles_in_step(n, j);
        for (int u = 0; u < nt; ++u) {
          const uint32_t p_addr = ptx::smem_u32(s.p[u]);
          const uint32_t v_addr = ptx::smem_u32(s.v[vs][u]);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_f8_ss(tO, ptx::sdesc_sw128(p_addr + 32 * kk, 16, 1024),
                           ptx::sdesc_sw128(v_addr + 4096 * kk, 8192, 1024), IDESC_PV,
                           (j > 0 || u > 0 || kk > 0) ? 1u : 0u);
        }
        ptx::mma_commit(&s.v_empty[vs]);
        ptx::mma_commit(&s.o_done);
      }
      if (!ok) break;
      g += nsteps;
      ++qk;
    } else if (k >= 1 && !attn::wait_bar(p, s, &s.o_empty, (k - 1) & 1)) {
      ok = false;
      break;
    }
    ptx::mbar_arrive(&s.task_empty[slot]);
  }
  ptx::mma_commit(&s.drain);
  attn::drain_bar(&s.drain, 0);
}

// ===================================================================================== softmax
// Warp (quarter, row block u, tile hf of the pair); a thread owns row r, columns
// [64 half, 64 half + 64) of tile hf.
__device__ __forceinline__ void run_softmax(const Params &p, Pipe &s, uint32_t tmem, int u,
                                            int hf) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quad = warp & 3;
  const int r = quad * 32 + u * 16 + (lane & 15);
  const int half = lane >> 4;
  const int col0 = half * 64;
  const uint32_t lanes = (uint32_t)(quad * 32 + u * 16) << 16;
  const uint32_t tS = tmem + lanes + S_COL + 128u * hf;
  const uint32_t tO = tmem + lanes + O_COL + 64u * hf;  // this warp's 64 columns of O
  uint8_t *prow = s.p[hf] + (r >> 3) * 1024 + (r & 7) * 128;
  // the exchange barrier of this row block completes once per step and once per task
  // (epilogue): before step j of task k its phase count is g + k + j
  const int xb = quad * 2 + u;
  int k = 0;
  uint32_t g = 0;
  for (;; ++k) {
    const int slot = k & 1;
    if (!attn::wait_bar_warp(p, s, &s.task_full[slot], (k >> 1) & 1)) break;
    const TaskInfo &ti = s.info[slot];
    const int n = ti.n;
    if (n < 0) break;
    const int nsteps = steps_of(n);
    const int t_hidden = n - 2;  // list tiles t >= n - 2 may hold hidden keys
    float row_scale;
    int causal_lim;
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
    const float rs_abs = fmaxf(fabsf(row_scale), 1e-30f);
    const uint64_t rs2 = ptx::pk(rs_abs, rs_abs);
    float m = -INFINITY, l = 0.f;  // l: this thread's share of the row sum
    const bool load_max = !p.k_per_token && !any_neg;
    bool ok = true;
    for (int j = 0; j < nsteps; ++j) {
      const uint32_t gs = g + j;
      // this warp's list tile; an odd last step has no second tile (t = n), which is run as a
      // tile whose keys are all hidden: its S columns hold a stale product that is masked to
      // -inf, so it adds nothing, and its P tile is not read by that step's PV
      const int t = 2 * j + hf;
      if (!attn::wait_bar_warp(p, s, &s.s_full, gs & 1)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      uint32_t x[2][32];
      float mx;
      ptx::tmem_ld16x2_64_max<64>(tS, x[0], x[1], mx);
      ptx::tmem_ld_wait(x[0]);
      ptx::reg_fence(x[1]);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&s.s_empty);
      if (p.k_per_token) {
        const int ds = gs % RING;
        if (!__all_sync(0xffffffffu, attn::wait_bar(p, s, &s.kd_full[ds], (gs / RING) & 1))) {
          ok = false;
          break;
        }
        const ulonglong2 *kd4 =
            reinterpret_cast<const ulonglong2 *>(&s.kd[ds][hf][kd_index(col0)]);
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int jj = 0; jj < 32; jj += 4) {
            const ulonglong2 kv = kd4[(c * 32 + jj) >> 2];
            float a0, a1, a2, a3;
            ptx::upk(ptx::mul2(ptx::pk(u2f(x[c][jj]), u2f(x[c][jj + 1])), kv.x), a0, a1);
            ptx::upk(ptx::mul2(ptx::pk(u2f(x[c][jj + 2]), u2f(x[c][jj + 3])), kv.y), a2, a3);
            x[c][jj] = f2u(a0);
            x[c][jj + 1] = f2u(a1);
            x[c][jj + 2] = f2u(a2);
            x[c][jj + 3] = f2u(a3);
          }
      }
      {
        if (any_neg) {
          const uint32_t flip = neg_scale ? 0x80000000u : 0u;
#pragma unroll
          for (int c = 0; c < 2; ++c)
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) x[c][jj] ^= flip;
        }
        if (t >= t_hidden) {
          const int tile = (t == t_hidden) ? ti.tail0 : ti.tail1;
          int lim = ti.kv_len - tile * TILE;
          if (p.causal) lim = min(lim, causal_lim - tile * TILE + 1);
          lim -= col0;
          if (t >= n) lim = 0;  // the missing second tile of an odd last step
          if (__any_sync(0xffffffffu, lim < 64)) {
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int jj = 0; jj < 32; ++jj)
                if (c * 32 + jj >= lim) x[c][jj] = f2u(-INFINITY);
          }
        }
        if (!(load_max && t < t_hidden)) {
          float a0 = -INFINITY, a1 = -INFINITY, a2 = -INFINITY, a3 = -INFINITY;
#pragma unroll
          for (int jj = 0; jj < 32; jj += 4) {
            a0 = ptx::max3(a0, u2f(x[0][jj]), u2f(x[0][jj + 1]));
            a1 = ptx::max3(a1, u2f(x[0][jj + 2]), u2f(x[0][jj + 3]));
            a2 = ptx::max3(a2, u2f(x[1][jj]), u2f(x[1][jj + 1]));
            a3 = ptx::max3(a3, u2f(x[1][jj + 2]), u2f(x[1][jj + 3]));
          }
          mx = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3));
        }
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));  // the row of this tile
      // the pair's row maximum: publish this tile's, meet the other tile's warp at xbar
      if (lane < 16) s.xmax[gs & 1][hf][r] = mx;
      ptx::mbar_arrive(&s.xch[xb]);
      // an inline wait: the S values are live here, and an out-of-line call would spill them
      if (!__all_sync(0xffffffffu, attn::wait_bar(p, s, &s.xch[xb], (gs + k) & 1))) {
        ok = false;
        break;
      }
      mx = fmaxf(mx, s.xmax[gs & 1][hf ^ 1][r]);
      const float m_new = fmaxf(m, mx * rs_abs);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ptx::ex2_approx(m - m_use);
      const uint64_t b2 = ptx::pk(p.log2_pscale - m_use, p.log2_pscale - m_use);
      uint32_t packed[16];
      float psum;
      {
        uint64_t acc0 = 0, acc1 = 0;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int jj = 0; jj < 32; jj += 4) {
            float e0, e1, e2, e3;
            ptx::upk(ptx::fma2(ptx::pk(u2f(x[c][jj]), u2f(x[c][jj + 1])), rs2, b2), e0, e1);
            ptx::upk(ptx::fma2(ptx::pk(u2f(x[c][jj + 2]), u2f(x[c][jj + 3])), rs2, b2), e2, e3);
            const float p0 = ptx::ex2_approx(e0), p1 = ptx::ex2_approx(e1);
            const float p2 = ptx::ex2_approx(e2), p3 = ptx::ex2_approx(e3);
            acc0 = ptx::add2(acc0, ptx::pk(p0, p1));
            acc1 = ptx::add2(acc1, ptx::pk(p2, p3));
            packed[(c * 32 + jj) >> 2] = ptx::cvt_e4m3x4(p0, p1, p2, p3);
          }
        float s0, s1, s2, s3;
        ptx::upk(acc0, s0, s1);
        ptx::upk(acc1, s2, s3);
        psum = (s0 + s1) + (s2 + s3);
      }
      l = alpha * l + psum;
      m = m_new;
      if (gs > 0) {
        // PV of the previous step done: the P tiles may be overwritten, O is stable
        if (!attn::wait_bar_warp(p, s, &s.o_done, (gs - 1) & 1)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4 *>(prow + (((4 * half + q) ^ (r & 7)) << 4)) =
            make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
      ptx::fence_proxy_async_smem();
      if (j > 0 && !__all_sync(0xffffffffu, alpha == 1.f)) {
        // O *= alpha on this thread's 32 of the warp's 64 columns
        const uint64_t a2 = ptx::pk(alpha, alpha);
        uint32_t o[32];
        ptx::tmem_ld16x2_32<32>(tO, o);
        ptx::tmem_ld_wait(o);
#pragma unroll
        for (int jj = 0; jj < 32; jj += 2) {
          float a, b3;
          ptx::upk(ptx::mul2(ptx::pk(u2f(o[jj]), u2f(o[jj + 1])), a2), a, b3);
          o[jj] = f2u(a);
          o[jj + 1] = f2u(b3);
        }
        ptx::tmem_st16x2_32<32>(tO, o);
        ptx::tmem_st_wait();
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&s.p_full);
      if (p.k_per_token) ptx::mbar_arrive(&s.kd_empty[gs % RING]);
    }
    if (!ok) break;
    // ------------------------------------------------------------------------- epilogue
    const int h = ti.h, qt = ti.qt;
    const bool row_ok = r < min(TILE, ti.q_len - qt * TILE);
    const int tok = ti.q0 + qt * TILE + r;
    const int g_kv = h / p.G;
    // the row sum: this tile's two column halves, then the other tile's warp
    float lt = l + __shfl_xor_sync(0xffffffffu, l, 16);
    if (lane < 16) s.xsum[hf][r] = lt;
    ptx::mbar_arrive(&s.xch[xb]);
    if (!attn::wait_bar_warp(p, s, &s.xch[xb], (g + nsteps + k) & 1)) break;
    const float l_row = lt + s.xsum[hf ^ 1][r];
    if (nsteps > 0) {
      if (!attn::wait_bar_warp(p, s, &s.o_done, (g + nsteps - 1) & 1)) break;
      ptx::tc_fence_after();
    }
    const bool seen = m != -INFINITY && l_row > 0.f;
    const float vd = p.v_per_head ? p.v_descale[g_kv] : p.v_descale[0];
    const float osc = seen ? vd / l_row : 0.f;
    uint32_t o[32];
    if (nsteps > 0) {
      ptx::tmem_ld16x2_32<32>(tO, o);
      ptx::tmem_ld_wait(o);
    } else {
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) o[jj] = 0u;
    }
    const uint64_t osc2 = ptx::pk(osc, osc);
    uint32_t w[16];
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      float a, b3;
      ptx::upk(ptx::mul2(ptx::pk(u2f(o[2 * jj]), u2f(o[2 * jj + 1])), osc2), a, b3);
      __nv_bfloat162 v2 = __floats2bfloat162_rn(a, b3);
      w[jj] = *reinterpret_cast<uint32_t *>(&v2);
    }
    if (row_ok) {
      uint4 *orow = reinterpret_cast<uint4 *>(p.out + ((size_t)tok * p.N1 + h) * HEAD_DIM +
                                              64 * hf + 32 * half);
#pragma unroll
      for (int q = 0; q < 4; ++q)
        orow[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    }
    ptx::tc_fence_before();
    ptx::mbar_arrive(&s.o_empty);
    if (hf == 0 && half == 0 && row_ok && p.lse) {
      p.lse[(size_t)h * p.T + tok] = seen ? (m + __log2f(l_row)) * 0.69314718055994531f -
                                                p.ln_pscale
                                          : -3.402823466e38f;
    }
    ptx::mbar_arrive(&s.task_empty[slot]);
    g += nsteps;
  }
}

__global__ void __launch_bounds__(NTHREADS, 1)
    bsa_attention_wide_kernel(const __grid_constant__ Params p,
                              const __grid_constant__ CUtensorMap tmap_q,
                              const __grid_constant__ CUtensorMap tmap_k,
                              const __grid_constant__ CUtensorMap tmap_v) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  Smem &sm = *reinterpret_cast<Smem *>(base);
  Pipe &s = sm.pipe;
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&s.task_full[i], 1);
      ptx::mbar_init(&s.task_empty[i], NSOFT + 1);  // the softmax threads + the MMA thread
    }
    ptx::mbar_init(&s.q_full, 1);
    ptx::mbar_init(&s.q_empty, 1);
    for (int i = 0; i < RING; ++i) {
      ptx::mbar_init(&s.k_full[i], 1);
      ptx::mbar_init(&s.k_empty[i], 1);
      ptx::mbar_init(&s.v_full[i], 1);
      ptx::mbar_init(&s.v_empty[i], 1);
      ptx::mbar_init(&s.kd_full[i], 1);
      ptx::mbar_init(&s.kd_empty[i], NSOFT);
    }
    ptx::mbar_init(&s.s_full, 1);
    ptx::mbar_init(&s.s_empty, NSOFT);
    ptx::mbar_init(&s.p_full, NSOFT);
    ptx::mbar_init(&s.o_done, 1);
    ptx::mbar_init(&s.o_empty, NSOFT);
    ptx::mbar_init(&s.drain, 1);
    for (int i = 0; i < 8; ++i) ptx::mbar_init(&s.xch[i], 64);  // the two warps of a row block
    s.abort_flag = 0;
    ptx::fence_mbarrier_init();
    ptx::prefetch_tmap(&tmap_q);
    ptx::prefetch_tmap(&tmap_k);
    ptx::prefetch_tmap(&tmap_v);
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
    if (warp == 0) {
      uint16_t *list = reinterpret_cast<uint16_t *>(base + sizeof(Smem));
      run_producer(p, s, list, &tmap_q, &tmap_k, &tmap_v);
    } else if (warp == 1 && (threadIdx.x & 31) == 0) {
      run_mma(p, s, sm.tmem_base);
    }
  } else {
    ptx::regs_inc<SOFTMAX_REGS>();
    const int wg = (warp >> 2) - 1;  // 0..3: row block wg % 2, tile wg / 2 of the pair
    run_softmax(p, s, sm.tmem_base, wg & 1, wg >> 1);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(sm.tmem_base, TMEM_COLS);
  }
}

}  // namespace attn_wide
}  // namespace bsa
