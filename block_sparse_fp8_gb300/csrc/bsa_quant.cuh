// The quantise step before the attention call: bf16 rows of 128 values -> e4m3 codes and an
// fp32 descale per row (FlashMLA page, section 量化 / 解量化的源码实现: scale = amax / 448,
// stored value e4m3(x / scale); optionally the scale rounded up to a power of two, the same
// section's cast to UE8M0), and the K/V append into the paged cache.
//
// HBM-bound.  A half-warp owns one 256-byte row: each lane loads 16 bytes (8 values), the row
// maximum combines in four shuffles, and each lane stores its 8 codes (8 bytes), so a warp
// reads 512 and writes 256 contiguous bytes per step.  The quotient is the correctly rounded
// fp32 x / scale (the code decision is taken in that precision on every side) and the
// conversion rounds to nearest even with saturation.
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "bsa_common.cuh"

namespace bsa {
namespace quant {

constexpr int THREADS = 256;  // 16 rows per block step

__device__ __forceinline__ void report_status(int *dev_status, int bits) {
  if (dev_status) atomicOr(dev_status, bits);
}

__device__ __forceinline__ void unpack8(const uint4 &w, float (&v)[8]) {
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(u[i] << 16);
    v[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
  }
}

// Largest |v| of the 128 values of the half-warp's row.
__device__ __forceinline__ float row_amax(const float (&v)[8]) {
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[i]));
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
  return a;
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}

// 8 codes of v / scale, the first value in the lowest byte.  The quotients are the correctly
// rounded fp32 quotients.  For a scale in [2^-90, 2^90] they come from Markstein's correction
// (P. Markstein, "Computation of elementary functions on the IBM RISC System/6000 processor",
// IBM J. Res. Dev. 34(1), 1990): with r the correctly rounded reciprocal of the scale,
// q0 = x*r, the remainder x - q0*scale (exact in one fma) and q = q0 + remainder*r rounded
// once give the correctly rounded x / scale whenever no intermediate leaves the normal range,
// which that scale range guarantees for every quotient that can round to a nonzero e4m3 code;
// three operations per value instead of a full division.  Other scales divide directly.
__device__ __forceinline__ uint2 codes8(const float (&v)[8], float scale) {
  float q[8];
  if (scale >= 0x1p-90f && scale <= 0x1p90f) {
    const float r = __frcp_rn(scale);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float q0 = v[i] * r;
      q[i] = fmaf(fmaf(-q0, scale, v[i]), r, q0);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(v[i], scale);
  }
  return make_uint2(e4m3x4(q[0], q[1], q[2], q[3]), e4m3x4(q[4], q[5], q[6], q[7]));
}

// The smallest power of two not below x (x > 0, finite, below 2^127), from its bits: a
// normal x with a zero fraction is one already, any other normal x goes to the next binade's
// first value; a subnormal x is its fraction times 2^-149, so the power of two is the
// fraction's, rounded up to the next power of two the same way.
__device__ __forceinline__ float pow2_ceil(float x) {
  const uint32_t b = __float_as_uint(x);
  const uint32_t e = b & 0x7f800000u, m = b & 0x007fffffu;
  if (m == 0u) return x;
  if (e != 0u) return __uint_as_float(e + 0x00800000u);
  return __uint_as_float((m & (m - 1u)) == 0u ? m : (1u << (32 - __clz(m))));
}

// descale of a row: amax / 448 (an fp32 quotient), or 1 for an all-zero row; with `ue8m0`
// rounded up to a power of two (so that a code times its descale is exact).
__device__ __forceinline__ float descale_of(float amax, bool ue8m0) {
  if (!(amax > 0.f)) return 1.f;
  const float d = __fdiv_rn(amax, 448.f);
  return ue8m0 ? pow2_ceil(d) : d;
}

__global__ void __launch_bounds__(THREADS) quantize_rows_kernel(const uint4 *__restrict__ x,
                                                                long long rows,
                                                                uint2 *__restrict__ codes,
                                                                float *__restrict__ descale,
                                                                bool ue8m0) {
  const int lane = threadIdx.x & 15;
  const long long step = (long long)gridDim.x * (THREADS / 16);
  // every lane runs the same number of iterations (the shuffles need the whole warp); each
  // iteration takes two rows, both loads in flight before either is used
  const long long first = (long long)blockIdx.x * (THREADS / 16) + (threadIdx.x >> 4);
  const long long iters = (rows + 2 * step - 1) / (2 * step);
  for (long long it = 0; it < iters; ++it) {
    const long long r0 = first + 2 * it * step, r1 = r0 + step;
    const bool live0 = r0 < rows, live1 = r1 < rows;
    const uint4 w0 = live0 ? x[r0 * 16 + lane] : make_uint4(0, 0, 0, 0);
    const uint4 w1 = live1 ? x[r1 * 16 + lane] : make_uint4(0, 0, 0, 0);
    float v[8];
    unpack8(w0, v);
    const float d0 = descale_of(row_amax(v), ue8m0);
    if (live0) {
      codes[r0 * 16 + lane] = codes8(v, d0);
      if (lane == 0) descale[r0] = d0;
    }
    unpack8(w1, v);
    const float d1 = descale_of(row_amax(v), ue8m0);
    if (live1) {
      codes[r1 * 16 + lane] = codes8(v, d1);
      if (lane == 0) descale[r1] = d1;
    }
  }
}

struct AppendParams {
  const uint4 *k_new, *v_new;
  const int *cu_new, *cache_len, *block_table;
  const float *k_scale, *v_scale;
  uint2 *k_pages, *v_pages;
  float *k_descale;
  int *dev_status;
  int B, N2, ps, num_pages, L, total_new;
  int k_per_token, v_per_head, kv_nhd;
  int k_ue8m0;  // per-token K descales rounded up to a power of two
};

// One warp per new token.  The token's first four heads of K and V are loaded before its
// page is looked up, so that the lookup's dependent reads (the sequence by binary search over
// cu_new, then the block table) overlap those loads; the two half-warps then take two heads at
// a time, four heads per batch of loads (deeper batches cost occupancy and measured slower).
constexpr int APPEND_PAIRS = 2;  // head pairs loaded per batch

__global__ void __launch_bounds__(THREADS) append_kv_kernel(const AppendParams p) {
  const int lane = threadIdx.x & 31, hl = lane & 15, hw = lane >> 4;
  const int warps = gridDim.x * (THREADS / 32);
  for (int tok = blockIdx.x * (THREADS / 32) + (threadIdx.x >> 5); tok < p.total_new;
       tok += warps) {
    uint4 wk[APPEND_PAIRS], wv[APPEND_PAIRS];
    auto load = [&](int g0) {
#pragma unroll
      for (int j = 0; j < APPEND_PAIRS; ++j) {
        const int g = g0 + 2 * j + hw;
        const long long r = (long long)tok * p.N2 + g;
        wk[j] = g < p.N2 ? p.k_new[r * 16 + hl] : make_uint4(0, 0, 0, 0);
        wv[j] = g < p.N2 ? p.v_new[r * 16 + hl] : make_uint4(0, 0, 0, 0);
      }
    };
    load(0);
    long long slot = 0;
    int pg = -1;
    if (lane == 0) {
      // sequence of the token: the last b with cu_new[b] <= tok
      int lo = 0, hi = p.B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.cu_new[mid] <= tok) lo = mid; else hi = mid - 1;
      }
      const long long pos = (long long)p.cache_len[lo] + (tok - p.cu_new[lo]);
      const long long lp = pos / p.ps;
      pg = (pos >= 0 && lp < p.L) ? p.block_table[(size_t)lo * p.L + lp] : -1;
      if (pg < 0 || pg >= p.num_pages) {
        report_status(p.dev_status, BSA_DEV_BAD_PAGE);
        pg = -1;
      } else {
        slot = pos % p.ps;
      }
    }
    pg = __shfl_sync(0xffffffffu, pg, 0);
    slot = __shfl_sync(0xffffffffu, slot, 0);
    if (pg < 0) continue;  // warp-uniform
    for (int g0 = 0; g0 < p.N2; g0 += 2 * APPEND_PAIRS) {
      if (g0 > 0) load(g0);
#pragma unroll
      for (int j = 0; j < APPEND_PAIRS; ++j) {
        const int g = g0 + 2 * j + hw;
        const bool live = g < p.N2;
        const long long dst = ((long long)pg * p.N2 + g) * p.ps + slot;  // K descale index
        const long long row = p.kv_nhd ? ((long long)pg * p.ps + slot) * p.N2 + g : dst;
        float v[8];
        unpack8(wk[j], v);
        // the shuffles of row_amax run on every lane, live or not
        const float amax = row_amax(v);
        if (live) {
          const float d = p.k_per_token ? descale_of(amax, p.k_ue8m0) : p.k_scale[0];
          p.k_pages[row * 16 + hl] = codes8(v, d);
          if (p.k_per_token && hl == 0) p.k_descale[dst] = d;
          unpack8(wv[j], v);
          p.v_pages[row * 16 + hl] = codes8(v, p.v_per_head ? p.v_scale[g] : p.v_scale[0]);
        }
      }
    }
  }
}

}  // namespace quant
}  // namespace bsa
