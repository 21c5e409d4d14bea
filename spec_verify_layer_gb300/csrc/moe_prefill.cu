// Prefill-width MoE layer (many token rows at once) for GB300 (sm_103a).
//
// The infero README ("Beyond plain text decode", MoE) routes prefill through a
// counting sort of the (token, expert) picks by expert followed by one GEMM per expert;
// this is that path on the same packed int4 weights as the verify-round kernel:
//   1 router     logits[t][e], fp32, the canonical order of the verify kernel (a warp
//                per 4 tokens x 4 experts, lane partials, xor tree)
//   2 top-k      a warp per token: k largest (logit desc, id asc), renormalised weights,
//                tokens per expert (atomic counts)
//   3 scan       exclusive prefixes of the counts and of the GEMM tiles per expert
//   4 scatter    every pick gets a slot in its expert's run (order inside a run is
//                free: each token's result does not depend on where it sits in a tile)
//   5 gate/up    per (expert, 64 tokens, 64 units) tile: mma.sync m16n8k16 bf16 with the
//                int4 codes turned into exact bf16 (n - 8), per-block fp32 scale, then
//                h' = w silu(g) v, stored as bf16 hi + lo in the down operand order
//   6 down       per (expert, 32 tokens, 128 output rows) tile: y = Wd h' (hi and lo
//                MMAs), fp32, to a per-pick buffer
//   7 combine    out[t] = sum over the token's picks in rank order (deterministic)
// Operands stream through a 3-stage cp.async ring in shared memory; packed blocks are
// read in the permuted order the packer wrote them (8 blocks = one 128-byte run).
#include <mutex>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int kPfThreads = 256;
constexpr int kPfWarps = kPfThreads / 32;
constexpr int kGuTok = 64;    // tokens per gate/up tile
constexpr int kGuUnits = 64;  // units (gate + up row pairs) per gate/up tile
constexpr int kDnTok = 32;    // tokens per down tile
constexpr int kDnRows = 128;  // output rows per down tile
constexpr int kStages = 3;
constexpr int kARows = 128;                       // A rows per tile, both GEMMs
constexpr int kACodes = kARows * 128;             // 8 blocks x 16 B per row
constexpr int kAScales = kARows * 16;             // 8 fp16 per row
constexpr int kBBytes = 32768;                    // 64 tokens x 256 bf16, or 32 tokens x 256 (hi, lo)
constexpr int kStageBytes = kACodes + kAScales + kBBytes;
constexpr int kPfSmem = kStages * kStageBytes;
constexpr unsigned kStatusBadSlot = 2u;
static_assert(kGuUnits * 2 == kARows && kDnRows == kARows, "one A tile shape");
static_assert(kGuTok * 256 * 2 == kBBytes && kDnTok * 256 * 4 == kBBytes, "one B stage size");

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Bank slot of expert e (the layer's expert -> slot table, if any); a slot outside the
// bank is reported and replaced by slot 0, so no read leaves the bank.
__device__ __forceinline__ int slot_of(const PrefillArgs& a, int e) {
  if (!a.slot) return e;
  const int s = __ldg(a.slot + e);
  if ((unsigned)s >= (unsigned)a.n_slots) {
    atomicOr(a.status, kStatusBadSlot);
    return 0;
  }
  return s;
}

// Tile index -> expert: the largest e with prefix[e] <= tile (prefix has E + 1 entries).
__device__ __forceinline__ int tile_expert(const int* prefix, int E, int tile) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(prefix + mid) <= tile) lo = mid;
    else hi = mid;
  }
  return lo;
}

// ---- 1 router: a warp per (4 tokens, 4 experts); the canonical order per logit ----
__global__ void __launch_bounds__(kPfThreads) k_pf_router(PrefillArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * 4, e0 = (blockIdx.y * kPfWarps + warp) * 4;
  if (e0 >= a.E) return;
  const int nt = min(4, a.T - t0), ne = min(4, a.E - e0);
  float p[4][4];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int e = 0; e < 4; ++e) p[r][e] = 0.f;
  for (int c = 0; c < a.H / 128; ++c) {
    const int h = 128 * c + 4 * lane;
    float xv[4][4], wv[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint2 u = (r < nt) ? __ldg(reinterpret_cast<const uint2*>(a.x + (size_t)(t0 + r) * a.H + h))
                               : make_uint2(0u, 0u);
      xv[r][0] = bf16_lo(u.x);
      xv[r][1] = bf16_hi(u.x);
      xv[r][2] = bf16_lo(u.y);
      xv[r][3] = bf16_hi(u.y);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float4 f = (e < ne) ? __ldg(reinterpret_cast<const float4*>(a.router + (size_t)(e0 + e) * a.H + h))
                                : make_float4(0.f, 0.f, 0.f, 0.f);
      wv[e][0] = f.x;
      wv[e][1] = f.y;
      wv[e][2] = f.z;
      wv[e][3] = f.w;
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int e = 0; e < 4; ++e) p[r][e] = __fmaf_rn(wv[e][j], xv[r][j], p[r][e]);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1)
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int e = 0; e < 4; ++e) p[r][e] = __fadd_rn(p[r][e], __shfl_xor_sync(0xffffffffu, p[r][e], o));
  if (lane == 0)
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (r < nt && e < ne) a.logits[(size_t)(t0 + r) * a.E + e0 + e] = p[r][e];
}

// ---- 2 top-k, renormalised weights and tokens per expert: a warp per token ----
__global__ void __launch_bounds__(kPfThreads) k_pf_topk(PrefillArgs a) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * kPfWarps + (threadIdx.x >> 5);
  if (t >= a.T) return;
  float my_l = 0.f;
  int my_id = 0;
  if (a.E <= 128)
    select_row<4>(a.logits + (size_t)t * a.E, a.E, a.k, lane, my_l, my_id);
  else
    select_row<16>(a.logits + (size_t)t * a.E, a.E, a.k, lane, my_l, my_id);
  // w_j = exp(l_j - l_1) / sum over the k picks (a warp sum: a fixed order per token)
  const float l1 = __shfl_sync(0xffffffffu, my_l, 0);
  const float ex = (lane < a.k) ? expf(my_l - l1) : 0.f;
  const float den = warp_sum(ex);
  if (lane < a.k) {
    const int p = t * a.k + lane;
    a.ids[p] = my_id;
    a.w[p] = __fdiv_rn(ex, den);
    atomicAdd(a.counts + my_id, 1);
  }
}

// ---- 3 prefixes (one CTA, one thread per expert, E <= 512) ----
__global__ void __launch_bounds__(512) k_pf_scan(PrefillArgs a) {
  __shared__ int s[3][512];
  const int e = threadIdx.x;
  const int c = (e < a.E) ? a.counts[e] : 0;
  int v[3] = {c, (c + kGuTok - 1) / kGuTok, (c + kDnTok - 1) / kDnTok};
#pragma unroll
  for (int q = 0; q < 3; ++q) s[q][e] = v[q];
  __syncthreads();
  for (int o = 1; o < 512; o <<= 1) {  // inclusive scans (Hillis-Steele)
    int add[3];
#pragma unroll
    for (int q = 0; q < 3; ++q) add[q] = (e >= o) ? s[q][e - o] : 0;
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 3; ++q) s[q][e] += add[q];
    __syncthreads();
  }
  if (e < a.E) {
    a.offs[e] = s[0][e] - v[0];
    a.cursor[e] = s[0][e] - v[0];
    a.tiles_gu[e] = s[1][e] - v[1];
    a.tiles_dn[e] = s[2][e] - v[2];
    if (a.user_counts) a.user_counts[e] = c;
  }
  if (e == a.E - 1) {
    a.offs[a.E] = s[0][e];
    a.tiles_gu[a.E] = s[1][e];
    a.tiles_dn[a.E] = s[2][e];
  }
}

// ---- 4 scatter: pick p = t k + j -> a slot of its expert's run ----
__global__ void __launch_bounds__(kPfThreads) k_pf_scatter(PrefillArgs a) {
  const int p = blockIdx.x * kPfThreads + threadIdx.x;
  if (p >= a.T * a.k) return;
  const int pos = atomicAdd(a.cursor + a.ids[p], 1);
  a.pos_tok[pos] = p / a.k;
  a.pos_pick[pos] = p;
  a.pick_pos[p] = pos;
}

// ---- 5 gate/up GEMM tiles ----
//
// A tile: 64 units of one expert = 128 packed rows (row 2u gate, 2u + 1 up) x one K
// chunk of 8 blocks (the 128-byte run holding logical blocks 8q..8q+7 of the row, in the
// row's permuted order).  MMA m-tile m = units 8m..8m+7, A row g = the gate row of unit
// 8m + g, row g + 8 = its up row: the lane holding a gate sum also holds the matching
// up sum.  B tile: 64 tokens x 256 activations, 16-byte pieces swizzled by token so a
// fragment load is conflict-free.  Warp w: m-tiles 2(w/2), 2(w/2)+1 x n-tiles 4(w%2) ..
// 4(w%2)+3.
__global__ void __launch_bounds__(kPfThreads, 1) k_pf_gateup(PrefillArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tile = blockIdx.x;
  if (tile >= a.tiles_gu[a.E]) return;
  const int e = tile_expert(a.tiles_gu, a.E, tile);
  const int p0 = a.offs[e] + (tile - a.tiles_gu[e]) * kGuTok;
  const int ntok = min(kGuTok, a.offs[e + 1] - p0);
  const int u0 = blockIdx.y * kGuUnits;
  const int H = a.H, NB = H >> 5, NBI = a.I >> 5;
  const int sl = slot_of(a, e);
  const uint8_t* codes = a.gu_nib + ((size_t)sl * a.I + u0) * 2 * NB * 16;
  const uint16_t* scales = a.gu_sc + ((size_t)sl * a.I + u0) * 2 * NB;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int wm = warp >> 1, wn = warp & 1;
  // this thread's B rows (token rows of x) for the staging copies: pieces tid + 256 i
  const int nq = NB / 8;

  auto load_stage = [&](int st, int q) {
    uint8_t* A = smem + st * kStageBytes;
    uint8_t* S = A + kACodes;
    uint8_t* B = S + kAScales;
#pragma unroll
    for (int i = 0; i < 4; ++i) {  // A codes: 128 rows x 8 pieces
      const int idx = tid + kPfThreads * i, r = idx >> 3, c = idx & 7;
      cp_async16(smem_addr(A + r * 128 + c * 16), codes + ((size_t)r * NB + 8 * q + c) * 16);
    }
    if (tid < kARows) cp_async16(smem_addr(S + tid * 16), scales + (size_t)tid * NB + 8 * q);
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // B: 64 tokens x 32 pieces of 8 activations
      const int idx = tid + kPfThreads * i, tk = idx >> 5, c = idx & 31;
      const int row = a.pos_tok[p0 + min(tk, ntok - 1)];  // tokens past the run repeat its last one
      cp_async16(smem_addr(B + tk * 512 + ((c ^ ((tk & 1) << 2)) * 16)), a.x + (size_t)row * H + 256 * q + 8 * c);
    }
  };

  float acc[2][4][4];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 4; ++ni)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[mi][ni][c] = 0.f;

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < nq) load_stage(s, s);
    cp_commit();
  }
  for (int q = 0; q < nq; ++q) {
    cp_wait<kStages - 2>();
    __syncthreads();
    if (q + kStages - 1 < nq) load_stage((q + kStages - 1) % kStages, q + kStages - 1);
    cp_commit();
    const uint8_t* A = smem + (q % kStages) * kStageBytes;
    const uint16_t* S = reinterpret_cast<const uint16_t*>(A + kACodes);
    const uint8_t* B = A + kACodes + kAScales;
#pragma unroll 2
    for (int b = 0; b < 8; ++b) {
      uint32_t bf[4][4];
#pragma unroll
      for (int ni = 0; ni < 4; ++ni) {
        const int tk = 8 * (4 * wn + ni) + g, c = 4 * b + t;
        bfrag_x(*reinterpret_cast<const uint4*>(B + tk * 512 + ((c ^ ((tk & 1) << 2)) * 16)), bf[ni]);
      }
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        const int u = 8 * (2 * wm + mi) + g, sw = b ^ ((u0 + u) & 7);
        uint32_t pg[4], pu[4];
        dq_word(*reinterpret_cast<const uint32_t*>(A + (2 * u) * 128 + sw * 16 + 4 * t), pg);
        dq_word(*reinterpret_cast<const uint32_t*>(A + (2 * u + 1) * 128 + sw * 16 + 4 * t), pu);
        const float sg = half_bits(S[(2 * u) * 8 + sw]), su = half_bits(S[(2 * u + 1) * 8 + sw]);
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          mma_bf16(d, pg[0], pu[0], pg[1], pu[1], bf[ni][0], bf[ni][1]);
          mma_bf16(d, pg[2], pu[2], pg[3], pu[3], bf[ni][2], bf[ni][3]);
          acc[mi][ni][0] = __fmaf_rn(sg, d[0], acc[mi][ni][0]);
          acc[mi][ni][1] = __fmaf_rn(sg, d[1], acc[mi][ni][1]);
          acc[mi][ni][2] = __fmaf_rn(su, d[2], acc[mi][ni][2]);
          acc[mi][ni][3] = __fmaf_rn(su, d[3], acc[mi][ni][3]);
        }
      }
    }
  }
  cp_wait<0>();
  // h' = w silu(g) v -> bf16 hi + lo at (position, intermediate index) in the down
  // pass's fragment order
#pragma unroll
  for (int mi = 0; mi < 2; ++mi) {
    const int i2 = u0 + 8 * (2 * wm + mi) + g, j = i2 & 31, e8 = j & 7;
#pragma unroll
    for (int ni = 0; ni < 4; ++ni)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int tk = 8 * (4 * wn + ni) + 2 * t + c;
        if (tk >= ntok) continue;
        const int pos = p0 + tk;
        const float gs = acc[mi][ni][c], vs = acc[mi][ni][2 + c];
        const float hh = __fmul_rn(__fdiv_rn(gs, __fadd_rn(1.f, expf(-gs))), vs);
        const float hw = __fmul_rn(a.w[a.pos_pick[pos]], hh);
        const __nv_bfloat16 hi = __float2bfloat16_rn(hw);
        const __nv_bfloat16 lo = __float2bfloat16_rn(__fsub_rn(hw, __bfloat162float(hi)));
        const size_t base = (((size_t)pos * NBI + (i2 >> 5)) * 4 + (j >> 3)) * 16 + 2 * (e8 & 3) + (e8 >> 2);
        a.hbuf[base] = __bfloat16_as_ushort(hi);
        a.hbuf[base + 8] = __bfloat16_as_ushort(lo);
      }
  }
}

// ---- 6 down GEMM tiles ----
//
// A tile: 128 output rows of one expert x one K chunk of 8 intermediate blocks; B tile:
// 32 positions x 256 intermediate values as (hi, lo) bf16 pieces, swizzled by position.
// Warp w: m-tiles 2(w/2), 2(w/2)+1 x n-tiles 2(w%2), 2(w%2)+1.  y -> ybuf[position][o].
__global__ void __launch_bounds__(kPfThreads, 1) k_pf_down(PrefillArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int tile = blockIdx.x;
  if (tile >= a.tiles_dn[a.E]) return;
  const int e = tile_expert(a.tiles_dn, a.E, tile);
  const int p0 = a.offs[e] + (tile - a.tiles_dn[e]) * kDnTok;
  const int ntok = min(kDnTok, a.offs[e + 1] - p0);
  const int o0 = blockIdx.y * kDnRows;
  const int H = a.H, NBI = a.I >> 5;
  const int sl = slot_of(a, e);
  // block-major down layout: block b of rows o0.. of the expert at (sl NBI + b) H + o0
  const uint8_t* codes = a.dn_nib + ((size_t)sl * NBI * H + o0) * 16;
  const uint16_t* scales = a.dn_sc + (size_t)sl * NBI * H + o0;
  const uint8_t* hb = reinterpret_cast<const uint8_t*>(a.hbuf);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
  const int wm = warp >> 1, wn = warp & 1;
  const int nq = NBI / 8;

  auto load_stage = [&](int st, int q) {
    uint8_t* A = smem + st * kStageBytes;
    uint8_t* S = A + kACodes;
    uint8_t* B = S + kAScales;
    // A: row r's block c of this stage at A + r 128 + (c ^ (r & 7)) 16 (eight rows of one
    // block fall in eight bank groups); S: scale of (r, c) at S[c 128 + r]
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int idx = tid + kPfThreads * i, c = idx >> 7, r = idx & 127;
      cp_async16(smem_addr(A + r * 128 + ((c ^ (r & 7)) * 16)), codes + ((size_t)(8 * q + c) * H + r) * 16);
    }
    if (tid < kARows) {
      const int c = tid >> 4, ch = tid & 15;
      cp_async16(smem_addr(S + c * 256 + ch * 16), scales + (size_t)(8 * q + c) * H + ch * 8);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // B: 32 positions x 64 pieces (8 blocks x 4 lanes x hi, lo)
      const int idx = tid + kPfThreads * i, tk = idx >> 6, c = idx & 63;
      const int pos = p0 + min(tk, ntok - 1);  // positions past the run repeat its last one
      cp_async16(smem_addr(B + tk * 1024 + ((c ^ (tk & 7)) * 16)), hb + ((size_t)pos * NBI + 8 * q) * 128 + c * 16);
    }
  };

  float acc[2][2][4];
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 2; ++ni)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[mi][ni][c] = 0.f;

#pragma unroll
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < nq) load_stage(s, s);
    cp_commit();
  }
  for (int q = 0; q < nq; ++q) {
    cp_wait<kStages - 2>();
    __syncthreads();
    if (q + kStages - 1 < nq) load_stage((q + kStages - 1) % kStages, q + kStages - 1);
    cp_commit();
    const uint8_t* A = smem + (q % kStages) * kStageBytes;
    const uint16_t* S = reinterpret_cast<const uint16_t*>(A + kACodes);
    const uint8_t* B = A + kACodes + kAScales;
#pragma unroll 2
    for (int b = 0; b < 8; ++b) {
      uint4 hv[2][2];
#pragma unroll
      for (int ni = 0; ni < 2; ++ni) {
        const int tk = 8 * (2 * wn + ni) + g, c = 8 * b + 2 * t;
        hv[ni][0] = *reinterpret_cast<const uint4*>(B + tk * 1024 + ((c ^ (tk & 7)) * 16));
        hv[ni][1] = *reinterpret_cast<const uint4*>(B + tk * 1024 + (((c + 1) ^ (tk & 7)) * 16));
      }
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        const int ra = 16 * (2 * wm + mi) + g, rb = ra + 8;
        const int sa = b ^ (ra & 7), sb = b ^ (rb & 7);
        uint32_t fa[4], fb[4];
        dq_word(*reinterpret_cast<const uint32_t*>(A + ra * 128 + sa * 16 + 4 * t), fa);
        dq_word(*reinterpret_cast<const uint32_t*>(A + rb * 128 + sb * 16 + 4 * t), fb);
        const float ska = half_bits(S[b * 128 + ra]), skb = half_bits(S[b * 128 + rb]);
#pragma unroll
        for (int ni = 0; ni < 2; ++ni) {
          const uint4 hi = hv[ni][0], lo = hv[ni][1];
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          mma_bf16(d, fa[0], fb[0], fa[1], fb[1], hi.x, hi.y);
          mma_bf16(d, fa[0], fb[0], fa[1], fb[1], lo.x, lo.y);
          mma_bf16(d, fa[2], fb[2], fa[3], fb[3], hi.z, hi.w);
          mma_bf16(d, fa[2], fb[2], fa[3], fb[3], lo.z, lo.w);
          acc[mi][ni][0] = __fmaf_rn(ska, d[0], acc[mi][ni][0]);
          acc[mi][ni][1] = __fmaf_rn(ska, d[1], acc[mi][ni][1]);
          acc[mi][ni][2] = __fmaf_rn(skb, d[2], acc[mi][ni][2]);
          acc[mi][ni][3] = __fmaf_rn(skb, d[3], acc[mi][ni][3]);
        }
      }
    }
  }
  cp_wait<0>();
#pragma unroll
  for (int mi = 0; mi < 2; ++mi)
#pragma unroll
    for (int ni = 0; ni < 2; ++ni)
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int tk = 8 * (2 * wn + ni) + 2 * t + c;
        if (tk >= ntok) continue;
        float* y = a.ybuf + (size_t)(p0 + tk) * H + o0 + 16 * (2 * wm + mi) + g;
        y[0] = acc[mi][ni][c];
        y[8] = acc[mi][ni][2 + c];
      }
}

// ---- 7 combine: out[t] = the token's picks' y in rank order ----
__global__ void __launch_bounds__(kPfThreads) k_pf_combine(PrefillArgs a) {
  const int H4 = a.H >> 2;
  const size_t i = (size_t)blockIdx.x * kPfThreads + threadIdx.x;
  if (i >= (size_t)a.T * H4) return;
  const int t = (int)(i / H4), o4 = (int)(i - (size_t)t * H4);
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < a.k; ++j) {
    const int pos = a.pick_pos[t * a.k + j];
    const float4 y = __ldcg(reinterpret_cast<const float4*>(a.ybuf + (size_t)pos * a.H) + o4);
    s.x = __fadd_rn(s.x, y.x);
    s.y = __fadd_rn(s.y, y.y);
    s.z = __fadd_rn(s.z, y.z);
    s.w = __fadd_rn(s.w, y.w);
  }
  reinterpret_cast<float4*>(a.out + (size_t)t * a.H)[o4] = s;
}

}  // namespace

int prefill_launch(const PrefillArgs& a, int* launches, void* stream) {
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(k_pf_gateup, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(k_pf_down, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
  });
  if (attr_err != cudaSuccess) return (int)attr_err;
  const int T = a.T, E = a.E, P = T * a.k;
  const int max_gu = (P + kGuTok - 1) / kGuTok + E, max_dn = (P + kDnTok - 1) / kDnTok + E;
  *launches = 0;
  cudaError_t e = cudaMemsetAsync(a.counts, 0, (size_t)E * 4, st);
  if (e != cudaSuccess) return (int)e;
  k_pf_router<<<dim3((T + 3) / 4, (E + 4 * kPfWarps - 1) / (4 * kPfWarps)), kPfThreads, 0, st>>>(a);
  k_pf_topk<<<(T + kPfWarps - 1) / kPfWarps, kPfThreads, 0, st>>>(a);
  k_pf_scan<<<1, 512, 0, st>>>(a);
  k_pf_scatter<<<(P + kPfThreads - 1) / kPfThreads, kPfThreads, 0, st>>>(a);
  k_pf_gateup<<<dim3(max_gu, a.I / kGuUnits), kPfThreads, kPfSmem, st>>>(a);
  k_pf_down<<<dim3(max_dn, a.H / kDnRows), kPfThreads, kPfSmem, st>>>(a);
  const size_t n4 = (size_t)T * (a.H / 4);
  k_pf_combine<<<(unsigned)((n4 + kPfThreads - 1) / kPfThreads), kPfThreads, 0, st>>>(a);
  *launches = 7;
  return (int)cudaGetLastError();
}

}  // namespace moe
