// Device helpers shared by the verify-round kernel (moe_verify.cu) and the
// prefill-width kernels (moe_prefill.cu).  Internal; not part of the public ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

namespace moe {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ float half_bits(uint16_t b) { return __half2float(__ushort_as_half(b)); }

// float -> unsigned key with the same order; -0 is first folded into +0 so that a
// signed-zero pair ties (and the lower id wins), as the definition asks.
__device__ __forceinline__ unsigned order_key(float v) {
  const unsigned u = __float_as_uint(__fadd_rn(v, 0.0f));
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(unsigned key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// True if (ka, ia) ranks before (kb, ib): larger key, then lower id.
__device__ __forceinline__ bool ranks_before(unsigned ka, int ia, unsigned kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// Top-k of one row of logits by one warp.  Lane l owns experts l + 32t (t < NE) as keys
// in registers; each of the k rounds takes the warp-wide best (redux.sync max on the
// key, then min on the id among equal keys) of the lanes' best keys and the owning lane
// drops it.  With up to 4 keys per lane they are sorted best-first once and a lane's
// best is its head; with more, a lane's best is found by a scan each round (keys only:
// a sorted network of 16 keys and ids spilled registers).  Lane j returns pick j
// (logit and id).
template <int NE>
__device__ __forceinline__ void select_row(const float* row, int E, int k, int lane, float& my_l,
                                           int& my_id) {
  unsigned kk[NE];
#pragma unroll
  for (int t = 0; t < NE; ++t) {
    const int e = lane + 32 * t;
    kk[t] = (e < E) ? order_key(__ldcg(row + e)) : 0u;  // (finite logits: keys >= 1)
  }
  if constexpr (NE <= 4) {
    // few keys per lane: sorted best-first once (ties: the lower id, i.e. the lower t,
    // first), then each round pops the winning lane's head
    int id[NE];
#pragma unroll
    for (int t = 0; t < NE; ++t) id[t] = lane + 32 * t;
#pragma unroll
    for (int size = 2; size <= NE; size <<= 1) {
#pragma unroll
      for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
        for (int i = 0; i < NE; ++i) {
          const int jj = i ^ stride;
          if (jj > i) {
            const bool up = (i & size) == 0;
            const bool sw = up ? ranks_before(kk[jj], id[jj], kk[i], id[i]) : ranks_before(kk[i], id[i], kk[jj], id[jj]);
            if (sw) {
              const unsigned tk = kk[i];
              kk[i] = kk[jj];
              kk[jj] = tk;
              const int ti = id[i];
              id[i] = id[jj];
              id[jj] = ti;
            }
          }
        }
      }
    }
    for (int j = 0; j < k; ++j) {
      const unsigned m = __reduce_max_sync(0xffffffffu, kk[0]);
      const unsigned win = __reduce_min_sync(0xffffffffu, kk[0] == m ? (unsigned)id[0] : 0xffffffffu);
      if ((unsigned)id[0] == win) {
#pragma unroll
        for (int t = 0; t + 1 < NE; ++t) {
          kk[t] = kk[t + 1];
          id[t] = id[t + 1];
        }
        kk[NE - 1] = 0u;
        id[NE - 1] = INT_MAX;
      }
      if (lane == j) {
        my_l = key_value(m);
        my_id = (int)win;
      }
    }
  } else {
    for (int j = 0; j < k; ++j) {
      unsigned best = kk[0];
      int bt = 0;
#pragma unroll
      for (int t = 1; t < NE; ++t)
        if (kk[t] > best) {
          best = kk[t];
          bt = t;
        }
      const unsigned mine = (unsigned)(lane + 32 * bt);
      const unsigned m = __reduce_max_sync(0xffffffffu, best);
      const unsigned win = __reduce_min_sync(0xffffffffu, best == m ? mine : 0xffffffffu);
      if (mine == win) {
#pragma unroll
        for (int t = 0; t < NE; ++t)
          if (t == bt) kk[t] = 0u;
      }
      if (lane == j) {
        my_l = key_value(m);
        my_id = (int)win;
      }
    }
  }
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// A 32-bit word of codes (eight nibbles, elements 0..7 of the word) -> four bf16 pairs
// (n - 8): (0, 4), (1, 5), (2, 6), (3, 7).
__device__ __forceinline__ void dq_word(uint32_t w, uint32_t (&p)[4]) {
  constexpr uint32_t M = 0x000F000Fu, C = 0x43004300u, B136 = 0x43084308u;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t v = ((w >> (4 * q)) & M) | C;  // 128 + n
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(p[q]) : "r"(v), "r"(B136));
  }
}

// Eight bf16 activations (elements 8t .. 8t+7 of a block) -> the same pairs.
__device__ __forceinline__ void bfrag_x(uint4 v, uint32_t (&b)[4]) {
  b[0] = __byte_perm(v.x, v.z, 0x5410);
  b[1] = __byte_perm(v.x, v.z, 0x7632);
  b[2] = __byte_perm(v.y, v.w, 0x5410);
  b[3] = __byte_perm(v.y, v.w, 0x7632);
}

// A warp's partial tiles ([2 n-tiles][16 rows][8 columns]) -> its scratch.
__device__ __forceinline__ void store_part(float* part, const float (&acc)[2][4], int g, int t) {
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    *reinterpret_cast<float2*>(part + nt * 128 + g * 8 + 2 * t) = make_float2(acc[nt][0], acc[nt][1]);
    *reinterpret_cast<float2*>(part + nt * 128 + (g + 8) * 8 + 2 * t) = make_float2(acc[nt][2], acc[nt][3]);
  }
}

}  // namespace moe
