// GB300 (sm_103a) kernel and C ABI of the MoE layer of a speculative-decoding verify
// round.  See include/moe_verify.h for the operation and the contract.
//
// A round of L layers is one persistent cooperative launch (one CTA per SM).  Two
// kernels share the router and routing phases:
//
// k_split (rounds of fewer than kMmaRows rows; the CUDA cores).  Per layer:
//   P1  router GEMV: this CTA's router rows (staged into shared memory while the
//       previous layer ran: they depend on no data), canonical fp32 order -> logits.
//   B1  (in its window: the slot table, this layer's activation digits and the previous
//       layer's output slice of this CTA)
//   P2  every CTA reads the logits and builds the same routing in shared memory:
//       per-row top-k (lower id wins ties), renormalised weights, the ascending expert
//       union U and, per union expert, the rows that picked it (CSR).
//   P3  the U * I/32 work units (union expert, 32-wide slice of the intermediate
//       dimension) are dealt to the CTAs heaviest first in snake order; a CTA streams
//       each unit's gate/up rows and down block column through shared memory, computes
//       the SwiGLU outputs of the slice and their share of the down product for every
//       output, and adds it as exact 2^32-scaled integers into the accumulators.
//   B3  (layer l+1's router waits for layer l's output, as a real decode would)
//
// k_round (wider rounds; the tensor cores): gate/up split by intermediate index, the
// SwiGLU outputs exchanged through the workspace under a second grid barrier, the down
// product by (expert, 16 output rows) units added as exact integers (see the section
// "Wide verify rounds" below).
//
// Expert dots on the CUDA cores are integer block dots: within a 32-element block,
// sum (n - 8) v over the nibble codes n and the activation v held in block fixed point
// (x: 16 bits in two byte digits; the SwiGLU output: 23 bits in three) is computed
// exactly with dp4a on the masked nibble bytes, then scaled once per block in fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int NT = 512;  // threads per CTA
constexpr int NW = NT / 32;
constexpr unsigned kStatusTimeout = 1u;
constexpr unsigned kStatusBadSlot = 2u;
constexpr unsigned long long kDefaultWaitNs = 2000000000ull;  // 2 s
// device waits count SM cycles: 2 cycles per requested ns bounds the wall time between
// ns (at ~2 GHz) and a few times ns at lower clocks
constexpr long long kCyclesPerNs = 2;
constexpr long long kDefaultWaitCycles = (long long)kDefaultWaitNs * kCyclesPerNs;
constexpr int kPhases = 13;  // phase stamps per layer when profiling (12 intervals)

struct LayerPtrs {
  const float* router;
  const uint8_t* gu_nib;
  const uint16_t* gu_sc;
  const uint8_t* dn_nib;
  const uint16_t* dn_sc;
  const int32_t* slot;  // expert -> bank slot, or null (slot = expert)
  int n_slots;
};

struct RoundArgs {
  int H, E, k, I, R, L;
  int Rmax;  // the handle's max_rows: the shared-memory plan is sized by it, not by R
  int route_only;
  int tail_rank;  // > 0: drop union experts every picking row has at 1-based rank >= it
  const uint16_t* x;  // [L][R][H] bf16 bits
  float* out;         // [L][R][H]
  int* stats;         // [L] |U| per layer, or null
  unsigned* bar;      // [0] barrier arrivals, [33] abort flag
  float* logits;      // [R][E]
  float* hbuf;        // [R*k][I] weighted SwiGLU outputs h' by CSR position (tensor-core rounds)
  unsigned long long* acc;  // [2][kSplitCopies][R][H] 2^32-scaled output accumulators (split rounds)
  int* user_ids;      // moe_route outputs (CTA 0 writes them)
  float* user_w;
  int* user_union;
  int* user_nunion;
  unsigned* status;
  long long wait_cycles;
  long long* phase_ts;  // [L][kPhases][grid] globaltimer stamps, or null
  LayerPtrs layer[kMaxLayers];
};

// ---------------------------------------------------------------------------------
// device helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}


__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(phase)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(phase)
      : "memory");
  return ok != 0;
}

// Waits for `phase` of the mbarrier for at most `limit` SM cycles; on giving up it
// raises the timeout bit of the status word and returns false.  The first poll does
// not block, so a bound of a few cycles gives up deterministically.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t phase, unsigned* status,
                                                  long long limit) {
  const long long t0 = clock64();
  if (mbar_test_wait(bar, phase)) return true;
  while (true) {
    if (clock64() - t0 > limit) {
      atomicOr(status, kStatusTimeout);
      return false;
    }
    if (mbar_try_wait(bar, phase)) return true;
  }
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ unsigned ld_relaxed(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---------------------------------------------------------------------------------
// grid barrier (all CTAs are co-resident: cooperative launch, one CTA per SM)

struct Sync {
  unsigned epoch = 0;
};

// Each CTA's thread 0 adds 1 to one counter with release semantics (ordering the CTA's
// earlier writes, published to it by the CTA barrier) and polls the counter with
// acquire loads until every CTA of this epoch has arrived.  On this GPU that costs
// about 1.2-1.4 us across both dies; a separate release flag, flag arrays, split
// counters and cluster-first hierarchies all measured slower.  Returns false if the
// round must be abandoned.
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Arrival half: the CTA's earlier writes are published by the CTA barrier and the
// release add.  Work that touches nothing other CTAs write may sit between the halves.
__device__ __forceinline__ void grid_arrive(const RoundArgs& a, Sync& sy) {
  __syncthreads();
  sy.epoch += 1;
  if (threadIdx.x == 0) red_release_add(a.bar, 1u);
}

__device__ bool grid_wait(const RoundArgs& a, const Sync& sy) {
  __shared__ int s_ok;
  if (threadIdx.x == 0) {
    const unsigned target = sy.epoch * gridDim.x;
    unsigned* abort_flag = a.bar + 33;
    int ok = 1;
    const long long t0 = clock64();
    while (ld_acquire(a.bar) < target) {
      if (ld_relaxed(abort_flag)) {
        ok = 0;
        break;
      }
      if (clock64() - t0 > a.wait_cycles) {
        atomicOr(a.status, kStatusTimeout);
        atomicExch(abort_flag, 1u);
        ok = 0;
        break;
      }
    }
    s_ok = ok;
  }
  __syncthreads();
  return s_ok != 0;
}

__device__ __forceinline__ bool grid_sync(const RoundArgs& a, Sync& sy) {
  grid_arrive(a, sy);
  return grid_wait(a, sy);
}

__device__ __forceinline__ void stamp(const RoundArgs& a, int l, int ph) {
  if (a.phase_ts && threadIdx.x == 0)
    a.phase_ts[((size_t)l * kPhases + ph) * gridDim.x + blockIdx.x] = clock64();
}

// ---------------------------------------------------------------------------------
// P1: router logits, one warp per expert, canonical order

// Router rows owned by this CTA: experts e = CTA + grid * q (q = 0, 1, ...).  They are
// staged into shared memory by one bulk copy per row, issued as soon as the previous
// layer's expert stream is done (router weights do not depend on any data).
__device__ __forceinline__ int router_rows_of_cta(int E) {
  return (E - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
}

__device__ void issue_router_rows(const RoundArgs& a, const float* router, float* s_rw,
                                  uint32_t bar) {
  const int n = router_rows_of_cta(a.E);
  if (n <= 0) return;
  const uint32_t row_bytes = (uint32_t)a.H * 4u;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_tx(bar, row_bytes * (uint32_t)n);
  for (int q = 0; q < n; ++q) {
    const int e = blockIdx.x + gridDim.x * q;
    bulk_g2s(smem_u32(s_rw + (size_t)q * a.H), router + (size_t)e * a.H, row_bytes, bar);
  }
}

// Lane l accumulates elements 128c + 4l + j for c ascending, then the xor-butterfly.
// The warps share out the (staged router row, activation row) pairs.
__device__ void router_phase(const RoundArgs& a, const uint16_t* x, const float* s_rw) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int NC = a.H >> 7;  // <= 16
  const int n = router_rows_of_cta(a.E);
  // (router row, activation row) pairs over the warps
  for (int pq = warp; pq < n * a.R; pq += NW) {
    const int q = pq / a.R, r = pq - q * a.R;
    const int e = blockIdx.x + gridDim.x * q;
    const float4* wr = reinterpret_cast<const float4*>(s_rw + (size_t)q * a.H) + lane;
    {
      const uint2* xr = reinterpret_cast<const uint2*>(x + (size_t)r * a.H) + lane;
      uint2 xv[16];
#pragma unroll
      for (int c = 0; c < 16; ++c)
        if (c < NC) xv[c] = __ldg(xr + 32 * c);
      float p = 0.f;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        if (c < NC) {
          const float4 w = wr[32 * c];
          p = __fmaf_rn(w.x, bf16_lo(xv[c].x), p);
          p = __fmaf_rn(w.y, bf16_hi(xv[c].x), p);
          p = __fmaf_rn(w.z, bf16_lo(xv[c].y), p);
          p = __fmaf_rn(w.w, bf16_hi(xv[c].y), p);
        }
      }
      p = warp_sum(p);
      if (lane == 0) a.logits[(size_t)r * a.E + e] = p;
    }
  }
}

// ---------------------------------------------------------------------------------
// P2: routing tables of one layer, built by every CTA in its shared memory

struct Tables {
  int* uni;      // [E] ascending union
  int* csr_off;  // [E+1] offsets into pair
  int* pair;     // [R*k] pair index p = r*k + j, grouped by union expert, rows ascending
  float* w;      // [R*k] renormalised weight of pair p
  int* n_union;  // [1]
  int* pos_ui;   // [R*k] union index of the expert at each CSR position
  int* pos_row;  // [R*k] row at each CSR position
  int* slot;     // [E] bank slot of each expert this layer
  int* pick_pos; // [R*k] CSR position of pick (r, j), or -1 if tail-skipped
};

// scratch (inside the staging area, free while routing): mask [E] (zeroed by the
// caller beforehand), off_e [E], ids [R*k], union index [E], best rank [E] (set to
// INT_MAX by the caller beforehand).
//
// Tail skip (Avalon README, "Numbers": experts that every token of a verification
// routes only at rank 7 or lower are skipped): with a.tail_rank = T > 0 an expert whose
// best 1-based rank over the rows that picked it is >= T leaves the union; its picks
// are not evaluated and the other weights are not renormalised.
// For the tensor-core kernel (wide != 0) it also cuts this CTA's share of the gate/up
// units into s_range[0..1] (first, end): units are shared out by work, a unit of an
// expert with R_e rows weighing ceil(R_e / 16); one row is an even split by count.  (The
// split kernel deals its units to the CTAs itself: split_unit_of.)
// One row without tail skip (E a power of two, 32 <= E <= 128; the counting work grows
// as E^2 and a larger E measured faster through the selection rounds): the whole
// routing by expert-parallel counting, no sequential rounds.  The rank of expert i is the number of
// experts that rank before it (larger logit, or equal logit and lower id), counted over
// quarters of the row by four threads; the k experts of rank < k are the picks (the
// same set and order as select_row), and a ballot over the experts in id order gives
// each pick its union index (the union is the k picks, ascending).  T.w[j] receives
// pick j's logit; softmax_one turns it into the weight.
__device__ __forceinline__ bool route_one_ok(const RoundArgs& a) {
  return a.R == 1 && a.tail_rank == 0 && a.E <= 128 && a.E >= 32 && (a.E & (a.E - 1)) == 0;
}

__device__ __forceinline__ int ranks_before_u(unsigned kj, int j, unsigned ki, int i) {
  return (kj > ki || (kj == ki && j < i)) ? 1 : 0;
}

__device__ void route_one(const RoundArgs& a, const Tables& T, unsigned* s_key, int* s_cnt, int* s_wc,
                          int layer) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, E = a.E, k = a.k;
  const int lgE = __ffs(E) - 1, QE = E >> 2;
  unsigned ki = 0;
  if (tid < E) {
    ki = order_key(__ldcg(a.logits + tid));
    s_key[tid] = ki;
  }
  __syncthreads();
  for (int task = tid; task < 4 * E; task += NT) {
    const int q = task >> lgE, i = task & (E - 1), j0 = q * QE;
    const unsigned kv = s_key[i];
    const uint4* row = reinterpret_cast<const uint4*>(s_key + j0);
    int cnt = 0;
    if (j0 + QE <= i || j0 > i) {
      // a quarter wholly below i ranks key j before i when kj >= ki, wholly above when
      // kj > ki (keys of finite logits are >= 1, so kj >= ki is kj > ki - 1)
      const unsigned th = (j0 > i) ? kv : kv - 1u;
#pragma unroll 8
      for (int j4 = 0; j4 < (QE >> 2); ++j4) {
        const uint4 v = row[j4];
        cnt += (v.x > th) + (v.y > th) + (v.z > th) + (v.w > th);
      }
    } else {
#pragma unroll 8
      for (int j4 = 0; j4 < (QE >> 2); ++j4) {
        const uint4 v = row[j4];
        const int j = j0 + 4 * j4;
        cnt += ranks_before_u(v.x, j, kv, i) + ranks_before_u(v.y, j + 1, kv, i) +
               ranks_before_u(v.z, j + 2, kv, i) + ranks_before_u(v.w, j + 3, kv, i);
      }
    }
    s_cnt[task] = cnt;
  }
  __syncthreads();
  const int rank = (tid < E) ? s_cnt[tid] + s_cnt[E + tid] + s_cnt[2 * E + tid] + s_cnt[3 * E + tid] : k;
  const bool picked = rank < k;
  const unsigned b = __ballot_sync(0xffffffffu, picked);
  if (lane == 0) s_wc[warp] = __popc(b);
  __syncthreads();
  int ui = __popc(b & ((1u << lane) - 1u));
  for (int w = 0; w < warp; ++w) ui += s_wc[w];
  if (picked && ui < k) {  // (exactly k are picked unless a logit is NaN, which is undefined)
    T.uni[ui] = tid;
    T.csr_off[ui] = ui;
    T.pos_ui[ui] = ui;
    T.pos_row[ui] = 0;
    T.pair[ui] = rank;
    T.pick_pos[rank] = ui;
    T.w[rank] = key_value(ki);
    if (blockIdx.x == 0) {
      if (a.user_ids) a.user_ids[rank] = tid;
      if (a.user_union) a.user_union[ui] = tid;
    }
  }
  if (tid == 0) {
    T.csr_off[k] = k;
    *T.n_union = k;
    if (blockIdx.x == 0) {
      if (a.user_nunion) *a.user_nunion = k;
      if (a.stats) a.stats[layer] = k;
    }
  }
  __syncthreads();
}

// Weights of route_one's picks (one warp): T.w[j] holds pick j's logit; w_j =
// exp(l_j - l_1) / sum over the k picks, the same warp sum as the general path.
__device__ void softmax_one(const RoundArgs& a, const Tables& T) {
  const int lane = threadIdx.x & 31, k = a.k;
  const float l = (lane < k) ? T.w[lane] : 0.f;
  const float l1 = __shfl_sync(0xffffffffu, l, 0);
  const float ex = (lane < k) ? expf(l - l1) : 0.f;
  const float den = warp_sum(ex);
  if (lane < k) {
    const float w = __fdiv_rn(ex, den);
    T.w[lane] = w;
    if (blockIdx.x == 0 && a.user_w) a.user_w[lane] = w;
  }
}

// Union, CSR tables and this CTA's unit range for rounds of at most 32 picks (no tail
// skip), by one warp: the picks, keyed (expert, row), are sorted across the lanes
// (bitonic network over xor partners); a pick that starts a run of one expert opens a
// union entry, and the ballot of those gives every pick its union index.  Same tables
// and the same unit cut as the general scan below.  s_ids holds the picks' experts.
__device__ void route_small(const RoundArgs& a, const Tables& T, const int* s_ids, int layer, int wide, int upe,
                            int* s_range) {
  const int lane = threadIdx.x & 31, k = a.k, P = a.R * k;
  constexpr unsigned FULL = 0xffffffffu;
  const bool live = lane < P;
  unsigned key = live ? ((unsigned)s_ids[lane] << 5) | (unsigned)(lane / k) : FULL;
  int pick = lane;
  // the network over the first NS lanes (NS = the power of two >= P) sorts them
  const int NS = P <= 8 ? 8 : (P <= 16 ? 16 : 32);
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
    if (size > NS) break;
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      const unsigned ok = __shfl_xor_sync(FULL, key, stride);
      const int op = __shfl_xor_sync(FULL, pick, stride);
      const bool keep_min = ((lane & size) == 0) == ((lane & stride) == 0);
      const bool sw = keep_min ? (ok < key) : (ok > key);
      key = sw ? ok : key;
      pick = sw ? op : pick;
    }
  }
  const int e = (int)(key >> 5), r = (int)(key & 31u);
  const unsigned prev = __shfl_up_sync(FULL, key, 1);
  const bool first = live && (lane == 0 || (prev >> 5) != (key >> 5));
  const unsigned fb = __ballot_sync(FULL, first);
  const int U = __popc(fb);
  const unsigned le = (lane == 31) ? FULL : ((2u << lane) - 1u);
  const int ui = __popc(fb & le) - 1;
  if (live) {
    T.pos_ui[lane] = ui;
    T.pos_row[lane] = r;
    T.pair[lane] = pick;
    T.pick_pos[pick] = lane;
  }
  if (first) {
    T.uni[ui] = e;
    T.csr_off[ui] = lane;
    if (blockIdx.x == 0 && a.user_union) a.user_union[ui] = e;
  }
  if (lane == 0) {
    T.csr_off[U] = P;
    *T.n_union = U;
    if (blockIdx.x == 0) {
      if (a.user_nunion) *a.user_nunion = U;
      if (a.stats) a.stats[layer] = U;
    }
  }
  if (!wide) return;  // (the split kernel deals its units itself)
  const int G = gridDim.x, c = blockIdx.x;
  if (a.R == 1) {
    const unsigned N = (unsigned)U * (unsigned)upe;
    if (lane == 0) {
      s_range[0] = (int)((c * N) / (unsigned)G);
      s_range[1] = (int)(((c + 1) * N) / (unsigned)G);
    }
    return;
  }
  __syncwarp();
  // union expert u = lane: its rows R_e and work weight, prefix over the union
  int wu = 0;
  if (lane < U) {
    const int re = T.csr_off[lane + 1] - T.csr_off[lane];
    wu = (re + 15) >> 4;
  }
  const int lw = upe * wu;
  int incw = lw;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int tw = __shfl_up_sync(FULL, incw, o);
    if (lane >= o) incw += tw;
  }
  const int wt_total = __shfl_sync(FULL, incw, 31), basew = incw - lw;
  const float wg = (float)wt_total / (float)G;
  const int tgt[2] = {c == 0 ? 0 : min((int)(wg * (float)c), wt_total),
                      c + 1 == G ? wt_total : min((int)(wg * (float)(c + 1)), wt_total)};
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    const bool here = lane < U && tgt[q] >= basew && tgt[q] < incw;
    const unsigned owner = __ballot_sync(FULL, here);
    int res = U * upe;
    if (owner) res = __shfl_sync(FULL, lane * upe + (tgt[q] - basew) / max(wu, 1), __ffs(owner) - 1);
    if (lane == 0) s_range[q] = res;
  }
}

__device__ int route_phase(const RoundArgs& a, const Tables& T, unsigned* s_mask, int* s_off_e,
                           int* s_ids, int* s_ui, int* s_rank, int layer, int wide, int upe, int* s_range) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, k = a.k, R = a.R;
  const bool small = R * k <= 32 && a.tail_rank == 0;
  // route_one's scratch: keys [E] (16-byte aligned: read as uint4), counts [4 E], warp sums
  unsigned* s_key = reinterpret_cast<unsigned*>((reinterpret_cast<uintptr_t>(s_rank + E) + 15) & ~(uintptr_t)15);
  if (route_one_ok(a)) {  // (weights: softmax_one, by the caller)
    route_one(a, T, s_key, reinterpret_cast<int*>(s_key + NT), reinterpret_cast<int*>(s_key + 5 * NT), layer);
    return k;
  }
  // rows: top-k, renormalised weights, row bits of each picked expert
  for (int r = warp; r < R; r += NW) {
    float my_l = 0.f;
    int my_id = 0;
    if (E <= 128)
      select_row<4>(a.logits + (size_t)r * E, E, k, lane, my_l, my_id);
    else  // E <= 512 (moe_create rejects more)
      select_row<16>(a.logits + (size_t)r * E, E, k, lane, my_l, my_id);
    // weights: exp(l_j - l_1) / sum over the k picks (a warp sum: a fixed order per row)
    const float l1 = __shfl_sync(0xffffffffu, my_l, 0);
    const float ex = (lane < k) ? expf(my_l - l1) : 0.f;
    const float den = warp_sum(ex);
    if (lane < k) {
      const float wj = __fdiv_rn(ex, den);
      const int p = r * k + lane;
      s_ids[p] = my_id;
      T.w[p] = wj;
      if (!small) atomicOr(&s_mask[my_id], 1u << r);
      if (a.tail_rank > 0) atomicMin(&s_rank[my_id], lane);
      if (blockIdx.x == 0) {
        if (a.user_ids) a.user_ids[p] = my_id;
        if (a.user_w) a.user_w[p] = wj;
      }
    }
  }
  __syncthreads();
  if (small) {
    if (warp == 0) route_small(a, T, s_ids, layer, wide, upe, s_range);
    __syncthreads();
    return *T.n_union;
  }
  // one warp: exclusive scans over e of (picked ? 1 : 0) and popc(mask) give the union
  // index and the CSR offset of every picked expert (lane l owns a contiguous range)
  if (warp == 0) {
    const int per = (E + 31) >> 5;  // <= 16
    const int e0 = lane * per, e1 = min(e0 + per, E);
    auto weight = [&](unsigned m) { return (__popc(m) + 15) >> 4; };
    int lf = 0, lc = 0, lw = 0;
    for (int e = e0; e < e1; ++e) {
      unsigned m = s_mask[e];
      if (m && a.tail_rank > 0 && s_rank[e] + 1 >= a.tail_rank) {
        m = 0u;  // tail-skipped: out of the union, its picks are dropped
        s_mask[e] = 0u;
      }
      lf += (m != 0u);
      lc += __popc(m);
      if (m) lw += upe * weight(m);
    }
    int incf = lf, incc = lc, incw = lw;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int tf = __shfl_up_sync(0xffffffffu, incf, o);
      const int tc = __shfl_up_sync(0xffffffffu, incc, o);
      const int tw = __shfl_up_sync(0xffffffffu, incw, o);
      if (lane >= o) {
        incf += tf;
        incc += tc;
        incw += tw;
      }
    }
    int basef = incf - lf, basec = incc - lc;
    // this CTA's unit range (the tensor-core kernel's gate/up units; the split kernel
    // deals its units itself): the targets t(c) ~ c W / G are computed the same way by
    // neighbouring CTAs (in fp32; monotone in c, t(0) = 0, t(G) = W), so the ranges
    // tile the units.
    if (wide) {
      const int G = gridDim.x, c = blockIdx.x;
      const int U = __shfl_sync(0xffffffffu, incf, 31);
      if (R == 1) {
        const unsigned N = (unsigned)U * (unsigned)upe;  // < 2^31 (U <= 512, upe <= 4096)
        if (lane == 0) {
          s_range[0] = (int)((c * N) / (unsigned)G);
          s_range[1] = (int)(((c + 1) * N) / (unsigned)G);
        }
      } else {
        const int wt_total = __shfl_sync(0xffffffffu, incw, 31), basew = incw - lw;
        const float wg = (float)wt_total / (float)G;
        const int tgt[2] = {c == 0 ? 0 : min((int)(wg * (float)c), wt_total),
                            c + 1 == G ? wt_total : min((int)(wg * (float)(c + 1)), wt_total)};
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const bool here = tgt[q] >= basew && tgt[q] < incw;
          int res = U * upe;
          if (here) {
            int cum = basew, ui = basef;
            for (int e = e0; e < e1; ++e) {
              const unsigned m = s_mask[e];
              if (!m) continue;
              const int w = weight(m), ew = upe * w;
              if (tgt[q] < cum + ew) {
                res = ui * upe + (tgt[q] - cum) / w;
                break;
              }
              cum += ew;
              ++ui;
            }
          }
          const unsigned owner = __ballot_sync(0xffffffffu, here);
          res = owner ? __shfl_sync(0xffffffffu, res, __ffs(owner) - 1) : U * upe;
          if (lane == 0) s_range[q] = res;
        }
      }
    }
    for (int e = e0; e < e1; ++e) {
      const unsigned m = s_mask[e];
      if (m) {
        s_off_e[e] = basec;
        s_ui[e] = basef;
        T.uni[basef] = e;
        T.csr_off[basef] = basec;
        if (blockIdx.x == 0 && a.user_union) a.user_union[basef] = e;
        ++basef;
        basec += __popc(m);
      }
    }
    if (lane == 31) {
      // the last lane's running totals are the union size and the pair count
      *T.n_union = basef;
      T.csr_off[basef] = basec;
      if (blockIdx.x == 0) {
        if (a.user_nunion) *a.user_nunion = basef;
        if (a.stats) a.stats[layer] = basef;
      }
    }
  }
  __syncthreads();
  for (int p = tid; p < R * k; p += NT) {
    const int e = s_ids[p], r = p / k;
    T.pick_pos[p] = -1;
    if (s_mask[e] == 0u) continue;  // (tail-skipped)
    const int pos = s_off_e[e] + __popc(s_mask[e] & ((1u << r) - 1u));
    T.pick_pos[p] = pos;
    T.pair[pos] = p;
    T.pos_row[pos] = r;
    T.pos_ui[pos] = s_ui[e];
  }
  __syncthreads();
  return *T.n_union;
}

// ---------------------------------------------------------------------------------
// Integer block dots.  A 32-element block of codes is four 32-bit words; word w holds
// elements 8w .. 8w+7, element 8w + 2j in the low nibble and 8w + 2j + 1 in the high
// nibble of byte j.  (w & 0x0F0F0F0F) gives the even elements' codes n as four bytes,
// (w & 0xF0F0F0F0) the odd elements' codes as 16 n, both without a shift.  The other
// operand is a block in fixed point: V_k = v_k 2^s as a signed integer of 16 bits (two
// byte digits, for the bf16 rows) or 24 bits (three digits, for the fp32 SwiGLU outputs),
// s chosen per block from its largest |v|; digit d of the elements in the same even/odd
// byte order.  dp4a then gives, exactly, per digit d:
//   A_d = sum over even k of n_k V_kd,   C_d = sum over odd k of 16 n_k V_kd,
// and 16 sum_k (n_k - 8) V_kd = 16 A_d + C_d - 128 sum_k V_kd  (= E_d, exact in int32).
// The block's sum (n - 8) v is 2^-s / 16 * sum_d 256^d E_d, formed in fp32.  A bf16 value
// within a factor 2^7 of its block's largest is exact in 16 bits; smaller ones are rounded
// to the block's 2^-s grid (an error below 2^-15 of the block maximum).  The 24-bit form
// keeps an fp32 value to 2^-22 of its block's maximum.
//
// Operand layouts (u32 words): digit word q = (d * 2 + parity) * 4 + w holds digit d of
// elements 8w + parity + 2j in byte j (j = 0..3).  Per block, after the digit words: the
// correction terms K_d = -128 sum_k V_kd (int) and the factor 2^-s / 16 (float).

__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Codes of one block as even / odd nibble bytes.
// round(v) for |v| < 2^22 on the FMA and integer pipes (the conversion instructions run
// on a slower shared pipe): adding 1.5 * 2^23, whose ulp is 1, rounds v to the nearest
// integer (ties to even, as __float2int_rn) into the low mantissa bits.  With v = x s
// for a power of two s, the fma rounds the exact product once: round(x s).
__device__ __forceinline__ int rint_small(float x, float s) {
  return __float_as_int(__fmaf_rn(x, s, 12582912.f)) - 0x4B400000;
}

struct NibBytes {
  uint32_t lo[4], hi[4];
};
__device__ __forceinline__ NibBytes nib_bytes(const uint4 nb) {
  NibBytes n;
  const uint32_t w[4] = {nb.x, nb.y, nb.z, nb.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    n.lo[i] = w[i] & 0x0F0F0F0Fu;
    n.hi[i] = w[i] & 0xF0F0F0F0u;
  }
  return n;
}

// A 16-bit operand block (two digits) in registers: digit words and K_0, K_1, factor.
struct Op16 {
  uint32_t d[16];
  int k0, k1;
  float f;
};
// A 24-bit operand block (three digits).
struct Op24 {
  uint32_t d[24];
  int k0, k1, k2;
  float f;
};

// sum over the block of (n - 8) v for a 16-bit operand.
// E_0 + 256 E_1 (16 times the block's sum, |.| < 2^28) is formed exactly in int32 and
// converted once: the same float as an fma of the two converted digit sums, which rounds
// the same exact integer once.  The correction terms seed the first digit's sum.
__device__ __forceinline__ float bdot16(const NibBytes& n, const Op16& x) {
  int a0 = 0, c0 = x.k0 + 256 * x.k1, a1 = 0, c1 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a0 = dp4a_uu(n.lo[i], x.d[i], a0);
    c0 = dp4a_uu(n.hi[i], x.d[4 + i], c0);
    a1 = dp4a_us(n.lo[i], x.d[8 + i], a1);
    c1 = dp4a_us(n.hi[i], x.d[12 + i], c1);
  }
  const int e = 16 * a0 + c0 + 256 * (16 * a1 + c1);
  return __fmul_rn(__int2float_rn(e), x.f);
}

// sum over the block of (n - 8) v for a 24-bit operand.
// E_0 + 256 E_1 (|.| < 2^29) exactly in int32 and converted once, as in bdot16; E_2
// joins in fp32.
__device__ __forceinline__ float bdot24(const NibBytes& n, const Op24& h) {
  int a0 = 0, c0 = h.k0 + 256 * h.k1, a1 = 0, c1 = 0, a2 = 0, c2 = h.k2;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a0 = dp4a_uu(n.lo[i], h.d[i], a0);
    c0 = dp4a_uu(n.hi[i], h.d[4 + i], c0);
    a1 = dp4a_uu(n.lo[i], h.d[8 + i], a1);
    c1 = dp4a_uu(n.hi[i], h.d[12 + i], c1);
    a2 = dp4a_us(n.lo[i], h.d[16 + i], a2);
    c2 = dp4a_us(n.hi[i], h.d[20 + i], c2);
  }
  const int e01 = 16 * a0 + c0 + 256 * (16 * a1 + c1), e2 = 16 * a2 + c2;
  return __fmul_rn(__fmaf_rn((float)e2, 65536.f, __int2float_rn(e01)), h.f);
}

// Byte j of digit word q for element e of a block: q = (d * 2 + (e & 1)) * 4 + (e >> 3),
// j = (e & 7) >> 1.
__device__ __forceinline__ int digit_word(int d, int e) { return (d * 2 + (e & 1)) * 4 + (e >> 3); }

// One block of 32 bf16 values (four 16-byte words) -> its 16-bit operand (digit words,
// K_0, K_1, factor).  s = 14 - e, e the unbiased exponent of the largest |value| (at
// least -113 so that 2^s stays a normal float): |V| < 2^15.
__device__ __forceinline__ void x_block_to_op16(const uint4 (&u)[4], Op16& op) {
  uint32_t v[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[4 * i] = u[i].x;
    v[4 * i + 1] = u[i].y;
    v[4 * i + 2] = u[i].z;
    v[4 * i + 3] = u[i].w;
  }
  uint32_t mx = 0u;
#pragma unroll
  for (int i = 0; i < 16; ++i) mx = max(mx, max(v[i] & 0x7FFFu, (v[i] >> 16) & 0x7FFFu));
  const int E = max((int)(mx >> 7), 14);  // biased exponent of the largest |x|
  const float scale = __int_as_float((268 - E) << 23);   // 2^(141 - E) = 2^(14 - e)
  // 2^(E - 145) = 2^-s / 16 (a subnormal float below E = 19)
  op.f = E >= 19 ? __int_as_float((E - 18) << 23) : __int_as_float(1 << (E + 4));
#pragma unroll
  for (int q = 0; q < 16; ++q) op.d[q] = 0u;
  int s0 = 0, s1 = 0;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const float xv = (e & 1) ? bf16_hi(v[e >> 1]) : bf16_lo(v[e >> 1]);
    const int X = rint_small(xv, scale);
    const int d0 = X & 0xFF, d1 = X >> 8;
    s0 += d0;
    s1 += d1;
    const int j = (e & 7) >> 1;
    op.d[digit_word(0, e)] |= (uint32_t)d0 << (8 * j);
    op.d[digit_word(1, e)] |= ((uint32_t)d1 & 0xFFu) << (8 * j);
  }
  op.k0 = -128 * s0;
  op.k1 = -128 * s1;
}

// This layer's rows as 16-bit operands in shared memory: s_xd [R][4][NB] uint4 (digit
// words 4c .. 4c+3 of block b at uint4 index c * NB + b, conflict-free for lane = block)
// and s_xk [R][NB] uint4 (K_0, K_1, factor bits, 0).  Done while the router barrier
// completes.
__device__ void stage_xdigits(const RoundArgs& a, const uint16_t* x, uint4* s_xd, uint4* s_xk) {
  const int NB = a.H >> 5;
  for (int idx = threadIdx.x; idx < a.R * NB; idx += NT) {
    const int r = idx / NB, b = idx - r * NB;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)r * a.H + 32 * b);
    uint4 u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) u[i] = __ldg(src + i);
    Op16 op;
    x_block_to_op16(u, op);
#pragma unroll
    for (int c = 0; c < 4; ++c)
      s_xd[((size_t)r * 4 + c) * NB + b] = make_uint4(op.d[4 * c], op.d[4 * c + 1], op.d[4 * c + 2], op.d[4 * c + 3]);
    s_xk[(size_t)r * NB + b] = make_uint4((uint32_t)op.k0, (uint32_t)op.k1, __float_as_uint(op.f), 0u);
  }
}

// The 16-bit operand of block blk of one row: from the staged digits (XS) or converted
// from the bf16 row in global memory (rows too many to stage).
template <bool XS>
__device__ __forceinline__ void load_xop(const RoundArgs& a, const uint16_t* x, const uint4* s_xd, const uint4* s_xk,
                                         int row, int blk, Op16& op) {
  const int NB = a.H >> 5;
  if (XS) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint4 v = s_xd[((size_t)row * 4 + c) * NB + blk];
      op.d[4 * c] = v.x;
      op.d[4 * c + 1] = v.y;
      op.d[4 * c + 2] = v.z;
      op.d[4 * c + 3] = v.w;
    }
    const uint4 k = s_xk[(size_t)row * NB + blk];
    op.k0 = (int)k.x;
    op.k1 = (int)k.y;
    op.f = __uint_as_float(k.z);
  } else {
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)row * a.H + 32 * blk);
    uint4 u[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) u[i] = __ldg(src + i);
    x_block_to_op16(u, op);
  }
}

// V values per lane (V a power of two <= 16) summed over the warp; value v ends in
// lanes [v 32/V, (v+1) 32/V).  Each value is summed over the same xor tree of lane bits
// 4..0 as warp_sum (only the operand order of commutative adds differs), so its result
// does not depend on the slot it travels in.
template <int V>
__device__ __forceinline__ float warp_sum_multi(float (&v)[V], int lane) {
  constexpr int LOGV = (V >= 16) ? 4 : (V >= 8) ? 3 : (V >= 4) ? 2 : (V >= 2) ? 1 : 0;
  static_assert((1 << LOGV) == V, "V must be a power of two <= 16");
#pragma unroll
  for (int s = 0; s < LOGV; ++s) {
    const int n = V >> s, o = 16 >> s;
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, o));
    }
  }
  float s = v[0];
#pragma unroll
  for (int o = 16 >> LOGV; o >= 1; o >>= 1) s = __fadd_rn(s, __shfl_xor_sync(0xffffffffu, s, o));
  return s;
}

// Leaving early: gives every copy still in flight a bounded chance to land (so no bulk
// copy targets shared memory of an exited CTA) and raises the abort flag.  Copies in
// flight are the pieces [k0, k1) of the current layer in a ring of `nslot` slots (piece
// k in slot (slot0 + k) % nslot, parity par0 ^ ((slot0 + k) / nslot & 1)) and the router
// rows.  Out of line: it never runs on the normal path.
__device__ __noinline__ void drain_and_abort(const RoundArgs& a, const uint64_t* bars, int nslot, unsigned slot0,
                                             unsigned par0, int k0, int k1, bool router_pend, uint32_t bar_router,
                                             unsigned ph_router) {
  if (threadIdx.x == 0) {
    for (int k = k0; k < k1; ++k) {
      const unsigned pos = slot0 + (unsigned)k;
      mbar_wait_bounded(smem_u32(bars + pos % (unsigned)nslot), par0 ^ ((pos / (unsigned)nslot) & 1u), a.status,
                        kDefaultWaitCycles);
    }
    if (router_pend) mbar_wait_bounded(bar_router, ph_router, a.status, kDefaultWaitCycles);
    atomicExch(a.bar + 33, 1u);
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------------
// Split-K rounds: the CUDA-core path (fewer than kMmaRows rows).
//
// Work unit (ui, s) = union expert ui, K-slice s: intermediate indices [32 s, 32 s + 32).
// Its bytes are the gate and up rows of those 32 indices (contiguous in the packed
// layout) and block s of every one of the expert's H down rows (contiguous in the
// block-major down layout): 3 * 32 * H / 2 code bytes and 3 * 32 * H / 16 scale bytes.
// The CTA that owns the unit computes, for every row r that picked the expert,
//   h'_r[i] = w_r silu(Wg[i] . x_r) (Wu[i] . x_r)         i in the slice
//   y_r[o]  = sum_{i in slice} Wd[o][i] h'_r[i]            every output o
// and adds y_r[o] * 2^32, rounded to an integer, into an int64 accumulator of row r.
// Integer adds are exact, so the accumulated value (and the fp32 output rounded from it)
// does not depend on the order of the adds, on how the units were shared out, or on the
// other rows of the round: a row's output is a function of that row alone, bit for bit.
// The adds go to one of kSplitCopies copies of the accumulator (by CTA), which keeps the
// number of adds that meet at one address small; after the layer's closing grid barrier
// each CTA sums the copies of its own output slice, writes the fp32 output and clears
// them.  No exchange of SwiGLU outputs between CTAs is needed, so a layer has two grid
// barriers (logits, layer end) instead of three, and the down products are computed
// while the stream is still running.
//
// Bytes are streamed as pieces of 9 H bytes into a ring of shared-memory slots (1-D bulk
// copies, one mbarrier per slot): four gate/up pieces (8 intermediate indices: 16 rows
// of H/2 code bytes, then their H/8-byte scale rows) and two down pieces (H/2 rows of
// one 16-byte block, then their fp16 scales) per unit, in unit order.

constexpr int kSplitCopies = kAccCopies;
constexpr int kSplitMaxSlots = 6;  // more slots measured slower (the ring crowds out L1)
constexpr int kGuPieces = 4;  // gate/up pieces per unit (8 intermediate indices each)
constexpr int kDnPieces = 2;  // down pieces per unit (H/2 output rows each)
constexpr int kPieces = kGuPieces + kDnPieces;
constexpr int kSplitPhases = 11;  // phase stamps per layer when profiling the split kernel

struct SplitPlan {
  size_t slot_bytes, ring, router, xd, xk, part, hd, uni, csr, pair, w, pos_ui, pos_row, slot, pick, order, nunion,
      misc, bars, total;
  int nslot, ng;
  bool x_staged, ok;
};

__host__ __device__ inline size_t up128(size_t x) { return (x + 127) & ~(size_t)127; }

// Shared-memory plan of the split kernel for R rows; the rows' operands are staged when
// they leave room for at least six slots.
__host__ __device__ inline SplitPlan split_plan(int H, int I, int E, int R, int k, int grid) {
  SplitPlan p{};
  const int NB = H >> 5;
  p.ng = (NB + 31) >> 5;
  p.slot_bytes = (size_t)9 * H;
  const size_t rk = (size_t)R * k;
  const size_t router = up128((size_t)((E + grid - 1) / grid) * H * 4);
  const size_t part = up128((size_t)64 * p.ng * R * 4);
  const size_t hd = up128((size_t)R * 28 * 4);
  const size_t tables = up128((size_t)E * 4) + up128((size_t)(E + 1) * 4) + 5 * up128(rk * 4) +
                        2 * up128((size_t)E * 4) + 128;
  const size_t misc = 256, bars = 256;
  const size_t limit = (size_t)225 * 1024;
  size_t fixed = router + part + hd + tables + misc + bars;
  const size_t xbytes = up128((size_t)R * H * 2) + up128((size_t)R * NB * 16);
  p.x_staged = fixed + xbytes + 6 * p.slot_bytes <= limit;
  if (p.x_staged) fixed += xbytes;
  int ns = fixed < limit ? (int)((limit - fixed) / p.slot_bytes) : 0;
  if (ns > kSplitMaxSlots) ns = kSplitMaxSlots;
  p.nslot = ns;
  size_t off = 0;
  p.ring = off;    off += (size_t)ns * p.slot_bytes;
  p.router = off;  off += router;
  p.xd = off;      off += p.x_staged ? up128((size_t)R * H * 2) : 0;
  p.xk = off;      off += p.x_staged ? up128((size_t)R * NB * 16) : 0;
  p.part = off;    off += part;
  p.hd = off;      off += hd;
  p.uni = off;     off += up128((size_t)E * 4);
  p.csr = off;     off += up128((size_t)(E + 1) * 4);
  p.pair = off;    off += up128(rk * 4);
  p.w = off;       off += up128(rk * 4);
  p.pos_ui = off;  off += up128(rk * 4);
  p.pos_row = off; off += up128(rk * 4);
  p.slot = off;    off += up128((size_t)E * 4);
  p.pick = off;    off += up128(rk * 4);
  p.order = off;   off += up128((size_t)E * 4);
  p.nunion = off;  off += 128;
  p.misc = off;    off += misc;
  p.bars = off;    off += bars;
  p.total = off;
  // routing scratch lives in the (then idle) ring: mask, offsets, ids, union index, best
  // rank, and the one-row counting path's keys, counts and warp sums
  const size_t scratch = ((size_t)4 * E + rk) * 4 + 16 + (size_t)(5 * NT + NW) * 4;
  p.ok = ns >= kGuPieces && (size_t)ns * p.slot_bytes >= scratch;
  return p;
}

// The split kernel's plan, in shared memory (written once per launch by thread 0).
__shared__ SplitPlan g_splan;

// Unit t of this CTA.  The union's units, heaviest first (experts by row count
// descending, then by union index, each expert's slices in order: s_order lists the
// union indices in that order; with one row every expert weighs the same and the order
// is the union's), are dealt out to the CTAs in snake order: round r gives
// one unit to every CTA, forward for even r and backward for odd r, so each CTA's load
// stays within about one light unit of the others' (a contiguous cut by work can put a
// whole heavy unit more on one CTA).  A unit is u = union index * NS + slice.
__device__ __forceinline__ int split_unit_of(int t, int NS, const int* s_order, int R) {
  const int G = gridDim.x, c = blockIdx.x;
  const int p = t * G + ((t & 1) ? G - 1 - c : c);
  const int q = p / NS;
  return (R > 1 ? s_order[q] : q) * NS + (p - q * NS);
}

// How many of the N units the deal gives this CTA.
__device__ __forceinline__ int split_unit_count(int N) {
  const int G = gridDim.x, c = blockIdx.x, full = N / G;
  return full + (((full & 1) ? G - 1 - c : c) < N - full * G ? 1 : 0);
}

// Piece pc of unit u -> ring slot dst (its completion counted on bar).
__device__ __forceinline__ void issue_piece(const RoundArgs& a, const LayerPtrs& W, const Tables& T, int NS, int u,
                                            int pc, uint8_t* dst, uint32_t bar, bool fence = true) {
  const size_t H = (size_t)a.H;
  const int ui = u / NS, s = u - ui * NS;
  const size_t sl = (size_t)T.slot[T.uni[ui]];
  const uint8_t* src_c;
  const uint8_t* src_s;
  if (pc < kGuPieces) {
    const size_t i0 = sl * (size_t)a.I + (size_t)s * 32 + (size_t)pc * 8;  // first intermediate index
    src_c = W.gu_nib + i0 * H;
    src_s = reinterpret_cast<const uint8_t*>(W.gu_sc) + i0 * (H / 8);
  } else {
    const size_t row0 = (sl * (size_t)NS + (size_t)s) * H + (size_t)(pc - kGuPieces) * (H / 2);
    src_c = W.dn_nib + row0 * 16;
    src_s = reinterpret_cast<const uint8_t*>(W.dn_sc) + row0 * 2;
  }
  if (fence) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_tx(bar, (uint32_t)(9 * H));
  bulk_g2s(smem_u32(dst), src_c, (uint32_t)(8 * H), bar);
  bulk_g2s(smem_u32(dst + 8 * H), src_s, (uint32_t)H, bar);
}

// ---- the split kernel's unit passes ----

// Gate/up of N consecutive rows rp0 .. rp0 + N - 1 of a gate/up piece (row rp of the
// piece = intermediate index i0 + rp / 2, gate for even rp, up for odd) for G activation
// rows: lane = hidden block b (32 kg + lane of the warp's K group), one block dot per row
// and activation row; v[g][j] = that block's contribution to row rp0 + j for activation
// g.  The codes and scales of all N rows are loaded before any is used.
template <int N, int G>
__device__ __forceinline__ void split_gu_rows(const uint8_t* piece, int H, int rp0, int b, bool valid,
                                              const Op16* xs, float (&v)[G][N]) {
  const int NB = H >> 5;
  const uint16_t* scales = reinterpret_cast<const uint16_t*>(piece + (size_t)8 * H);
  uint4 nb[N];
  float sc[N];
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const int rp = rp0 + j;
    // block b of the row of intermediate index i sits at b ^ (i & 7); i & 7 = (rp / 2) & 7
    const int pb = (b ^ ((rp >> 1) & 7)) & (valid ? 0xFFFF : 0);
    nb[j] = *reinterpret_cast<const uint4*>(piece + ((size_t)rp * NB + pb) * 16);
    sc[j] = valid ? half_bits(scales[rp * NB + pb]) : 0.f;
  }
#pragma unroll
  for (int j = 0; j < N; ++j) {
    const NibBytes n = nib_bytes(nb[j]);
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float t = __fmul_rn(sc[j], bdot16(n, xs[g]));
      v[g][j] = valid ? t : 0.f;  // (a lane past the row's blocks holds no operand)
    }
  }
}

// Reduces one activation row's N values over the warp and stores the row sums as
// partials of K group kg: s_part[((row0 + j) * NG + kg) * Rs + pr].
template <int N>
__device__ __forceinline__ void split_store_part(float (&v)[N], int lane, float* s_part, int row0, int NG, int kg,
                                                 int Rs, int pr) {
  const float s = warp_sum_multi<N>(v, lane);
  constexpr int LPV = 32 / N;
  if ((lane % LPV) == 0) s_part[((row0 + lane / LPV) * NG + kg) * Rs + pr] = s;
}

// The gate/up pass of one unit for this warp: rows [rb RPW, (rb + 1) RPW) of the unit's
// 64 (RPW = 4 NG, all in one piece), K group kg, every activation row of the expert (CSR
// positions p0 .. p0 + Re - 1) one after the other, four weight rows at a time (two rows
// at once, sharing the code bytes, measured slower: the operands no longer fit the
// registers).  XR: one row whose operand the caller holds in registers.
template <int NG, bool XR, bool XS>
__device__ __forceinline__ void split_gateup(const RoundArgs& a, const Tables& T, const uint8_t* piece, int rb,
                                             int kg, int p0, int Re, const Op16& xr, const uint4* s_xd,
                                             const uint4* s_xk, const uint16_t* x, float* s_part) {
  constexpr int RPW = 4 * NG;
  const int lane = threadIdx.x & 31, NB = a.H >> 5;
  const int b = 32 * kg + lane;
  const bool valid = b < NB;
  const int row0 = rb * RPW;
  // all of the warp's rows in one pass per activation row: one reduction, RPW
  // independent block dots
  if constexpr (XR) {
    float v[1][RPW];
    split_gu_rows<RPW, 1>(piece, a.H, row0 & 15, b, valid, &xr, v);
    split_store_part<RPW>(v[0], lane, s_part, row0, NG, kg, a.R, 0);
  } else {
    for (int pr = 0; pr < Re; ++pr) {
      Op16 xo[1];
      if (valid) load_xop<XS>(a, x, s_xd, s_xk, T.pos_row[p0 + pr], b, xo[0]);
      float v[1][RPW];
      split_gu_rows<RPW, 1>(piece, a.H, row0 & 15, b, valid, xo, v);
      split_store_part<RPW>(v[0], lane, s_part, row0, NG, kg, a.R, pr);
    }
  }
}

template <int NG, bool XS>
__device__ __forceinline__ void split_gateup_rows(const RoundArgs& a, const Tables& T, const uint8_t* piece, int rb,
                                                  int kg, int p0, int Re, const uint4* s_xd, const uint4* s_xk,
                                                  const uint16_t* x, float* s_part) {
  Op16 none;
  split_gateup<NG, false, XS>(a, T, piece, rb, kg, p0, Re, none, s_xd, s_xk, x, s_part);
}

// One row: this lane's block operand (row 0) comes from shared memory into registers
// once per unit and serves the warp's rows of the unit.
template <int NG>
__device__ __forceinline__ void split_gateup_one(const RoundArgs& a, const Tables& T, const uint8_t* piece, int rb,
                                                 int kg, int p0, const uint4* s_xd, const uint4* s_xk,
                                                 float* s_part) {
  const int NB = a.H >> 5, b = 32 * kg + (threadIdx.x & 31);
  Op16 xr;
  if (b < NB) {
    load_xop<true>(a, nullptr, s_xd, s_xk, 0, b, xr);
  } else {
#pragma unroll
    for (int q = 0; q < 16; ++q) xr.d[q] = 0u;
    xr.k0 = xr.k1 = 0;
    xr.f = 0.f;
  }
  split_gateup<NG, true, true>(a, T, piece, rb, kg, p0, 1, xr, s_xd, s_xk, nullptr, s_part);
}

// SwiGLU of one unit: warp per activation row (CSR position p0 + pr), lane = index i of
// the slice.  g and v add the K groups' partials in group order; h' = w silu(g) v.  The
// 32 values of h' go to s_hd[pr] as a 24-bit operand for the down pass: 24 digit words,
// then K_0, K_1, K_2 and the factor (28 words).
__device__ __forceinline__ void split_swiglu(const RoundArgs& a, const Tables& T, const float* s_part, int NG,
                                             int p0, int Re, uint32_t* s_hd) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int pr = warp; pr < Re; pr += NW) {
    float gs = s_part[((2 * lane) * NG) * a.R + pr], vs = s_part[((2 * lane + 1) * NG) * a.R + pr];
    for (int g = 1; g < NG; ++g) {
      gs = __fadd_rn(gs, s_part[((2 * lane) * NG + g) * a.R + pr]);
      vs = __fadd_rn(vs, s_part[((2 * lane + 1) * NG + g) * a.R + pr]);
    }
    const float hh = __fmul_rn(__fdiv_rn(gs, __fadd_rn(1.f, expf(-gs))), vs);
    const float hw = __fmul_rn(T.w[T.pair[p0 + pr]], hh);
    // s = 21 - e, e the unbiased exponent of the largest |h'| of the slice (at least
    // -105): |H| <= 2^22, three byte digits
    const unsigned mx = __reduce_max_sync(0xffffffffu, __float_as_uint(hw) & 0x7FFFFFFFu);
    const int E = max((int)(mx >> 23), 22);
    const float scale = __int_as_float((275 - E) << 23);  // 2^(148 - E)
    const int Hq = rint_small(hw, scale);
    const int d0 = Hq & 0xFF, d1 = (Hq >> 8) & 0xFF, d2 = Hq >> 16;
    uint8_t* row = reinterpret_cast<uint8_t*>(s_hd + pr * 28);
    const int j = (lane & 7) >> 1;
    row[digit_word(0, lane) * 4 + j] = (uint8_t)d0;
    row[digit_word(1, lane) * 4 + j] = (uint8_t)d1;
    row[digit_word(2, lane) * 4 + j] = (uint8_t)(d2 & 0xFF);
    const int s0 = (int)__reduce_add_sync(0xffffffffu, (unsigned)d0);
    const int s1 = (int)__reduce_add_sync(0xffffffffu, (unsigned)d1);
    const int s2 = (int)__reduce_add_sync(0xffffffffu, (unsigned)d2);
    if (lane == 0) {
      s_hd[pr * 28 + 24] = (uint32_t)(-128 * s0);
      s_hd[pr * 28 + 25] = (uint32_t)(-128 * s1);
      s_hd[pr * 28 + 26] = (uint32_t)(-128 * s2);
      // 2^(E - 152) = 2^-s / 16 (a subnormal float below E = 26)
      s_hd[pr * 28 + 27] = E >= 26 ? (uint32_t)((E - 25) << 23) : (1u << (E - 3));
    }
  }
}

// Fire-and-forget add at L2 (no value comes back, so the thread does not wait for it).
__device__ __forceinline__ void red_add_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("red.relaxed.gpu.global.add.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// This thread's down rows o = tid + NT j (j < kDnRowsPerThread) of a unit: codes and
// scales, loaded from the two down pieces before the SwiGLU barrier.
constexpr int kDnRowsPerThread = (kMaxHidden + NT - 1) / NT;
struct DnRows {
  uint4 nb[kDnRowsPerThread];
  float sc[kDnRowsPerThread];
};

__device__ __forceinline__ void load_dn_rows(int H, const uint8_t* dn0, const uint8_t* dn1, DnRows& d) {
  const int HH = H >> 1;
#pragma unroll
  for (int j = 0; j < kDnRowsPerThread; ++j) {
    const int o = (int)threadIdx.x + NT * j;
    if (o < H) {
      const uint8_t* pc = (o < HH) ? dn0 : dn1;
      const int ol = (o < HH) ? o : o - HH;
      d.nb[j] = *reinterpret_cast<const uint4*>(pc + (size_t)ol * 16);
      d.sc[j] = half_bits(reinterpret_cast<const uint16_t*>(pc + (size_t)8 * H)[ol]);
    } else {
      d.nb[j] = make_uint4(0u, 0u, 0u, 0u);
      d.sc[j] = 0.f;
    }
  }
}

// Down products of one unit for this thread's rows, every activation position of the
// expert in turn: y -> 2^32-scaled integers added into this CTA's accumulator copy.
__device__ __forceinline__ void split_down(const RoundArgs& a, const Tables& T, const DnRows& d, const uint32_t* s_hd,
                                           int p0, int Re, unsigned long long* acc_copy) {
  const int H = a.H;
  for (int pr = 0; pr < Re; ++pr) {
    Op24 hop;
    const uint4* src = reinterpret_cast<const uint4*>(s_hd + pr * 28);
#pragma unroll
    for (int c = 0; c < 6; ++c) {
      const uint4 v = src[c];
      hop.d[4 * c] = v.x;
      hop.d[4 * c + 1] = v.y;
      hop.d[4 * c + 2] = v.z;
      hop.d[4 * c + 3] = v.w;
    }
    const uint4 k = src[6];
    hop.k0 = (int)k.x;
    hop.k1 = (int)k.y;
    hop.k2 = (int)k.z;
    hop.f = __uint_as_float(k.w);
    unsigned long long* acc_row = acc_copy + (size_t)T.pos_row[p0 + pr] * H;
#pragma unroll
    for (int j = 0; j < kDnRowsPerThread; ++j) {
      const int o = (int)threadIdx.x + NT * j;
      if (o < H) {
        const float y = __fmul_rn(d.sc[j], bdot24(nib_bytes(d.nb[j]), hop));
        red_add_u64(acc_row + o, (unsigned long long)__float2ll_rn(y * 4294967296.0f));
      }
    }
  }
}

// This CTA's output slice [o0, o0 + no) of a finished layer: sum of the accumulator
// copies -> fp32 output; the copies are cleared for the next layer.  Threads from
// `first` on do it.
__device__ __forceinline__ void split_finish(const RoundArgs& a, int layer, int o0, int no, int first,
                                             int ncopies = kSplitCopies) {
  const size_t stride = (size_t)a.R * a.H;
  float* out = a.out + (size_t)layer * stride;
  unsigned long long* buf = a.acc + (size_t)(layer & 1) * kSplitCopies * stride;
  for (int i = (int)threadIdx.x - first; i < a.R * no; i += NT - first) {
    if (i < 0) break;
    const int r = i / no, o = o0 + (i - r * no);
    unsigned long long* p = buf + (size_t)r * a.H + o;
    unsigned long long s = 0ull;
    for (int c = 0; c < ncopies; ++c) s += __ldcg(p + c * stride);
    for (int c = 0; c < ncopies; ++c) __stcg(p + c * stride, 0ull);
    out[(size_t)r * a.H + o] = __fmul_rn(__ll2float_rn((long long)s), 0x1p-32f);
  }
}

__device__ __forceinline__ void split_stamp(const RoundArgs& a, int l, int ph) {
  if (a.phase_ts && threadIdx.x == 0)
    a.phase_ts[((size_t)l * kSplitPhases + ph) * gridDim.x + blockIdx.x] = clock64();
}

// This CTA's nu units of layer l (split_unit_of; their pieces 0 .. 6 nu - 1, piece k in
// ring slot (slot0 + k) % nslot with parity par0 ^ ((slot0 + k) / nslot & 1), the first
// n_init already issued); false (after draining) if a wait gave up.  Inlined: a call
// would save and restore the kernel's live registers through local memory, which the
// large shared-memory carve-out leaves little L1 for.
template <int NG, bool XR, bool XS>
__device__ __forceinline__ bool split_units(const RoundArgs& a, int l, unsigned char* smem, unsigned slot0,
                                            unsigned par0, int nu, int n_init, bool router_pend, uint32_t bar_router,
                                            unsigned ph_router) {
  const int tid = threadIdx.x, warp = tid >> 5;
  const int H = a.H, NS = a.I >> 5;
  const SplitPlan& P = g_splan;
  const int nslot = P.nslot;
  auto slot_of = [&](int k) { return (int)((slot0 + (unsigned)k) % (unsigned)nslot); };
  auto par_of = [&](int k) { return par0 ^ (((slot0 + (unsigned)k) / (unsigned)nslot) & 1u); };
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bars);
  uint8_t* ring = smem + P.ring;
  const uint4* s_xd = reinterpret_cast<const uint4*>(smem + P.xd);
  const uint4* s_xk = reinterpret_cast<const uint4*>(smem + P.xk);
  float* s_part = reinterpret_cast<float*>(smem + P.part);
  uint32_t* s_hd = reinterpret_cast<uint32_t*>(smem + P.hd);
  const Tables T{reinterpret_cast<int*>(smem + P.uni),     reinterpret_cast<int*>(smem + P.csr),
                 reinterpret_cast<int*>(smem + P.pair),    reinterpret_cast<float*>(smem + P.w),
                 reinterpret_cast<int*>(smem + P.nunion),  reinterpret_cast<int*>(smem + P.pos_ui),
                 reinterpret_cast<int*>(smem + P.pos_row), reinterpret_cast<int*>(smem + P.slot),
                 reinterpret_cast<int*>(smem + P.pick)};
  const int* s_order = reinterpret_cast<const int*>(smem + P.order);
  const LayerPtrs& W = a.layer[l];
  const uint16_t* x = a.x + (size_t)l * a.R * H;
  // layer l adds into accumulator buffer l & 1, copy blockIdx % kSplitCopies
  unsigned long long* acc_copy = a.acc + ((size_t)(l & 1) * kSplitCopies + blockIdx.x % kSplitCopies) * a.R * H;
  const int npieces = nu * kPieces;
  int issued = n_init;  // pieces of this layer issued so far (thread 0's count, uniform)
  int consumed = 0;
  const int rb = warp / NG, kg = warp % NG;
  const int my_piece = (rb * 4 * NG) >> 4;  // the gate/up piece holding this warp's rows
  bool stamped = false;
  for (int t = 0; t < nu; ++t) {
    const int ui = split_unit_of(t, NS, s_order, a.R) / NS;
    const int p0 = T.csr_off[ui], Re = T.csr_off[ui + 1] - p0;
    if (t + 1 == nu && t > 0) split_stamp(a, l, 6);
    // ---- gate/up: each warp waits for its own piece ----
    {
      const int J = t * kPieces + my_piece;
      bool ok = mbar_wait_bounded(smem_u32(bars + slot_of(J)), par_of(J), a.status, a.wait_cycles);
      if (ok) {
        if (!stamped && warp == 0) {
          split_stamp(a, l, 5);
          if (nu == 1) split_stamp(a, l, 6);
          stamped = true;
        }
        if (XR)
          split_gateup_one<NG>(a, T, ring + (size_t)slot_of(J) * P.slot_bytes, rb, kg, p0, s_xd, s_xk, s_part);
        else
          split_gateup_rows<NG, XS>(a, T, ring + (size_t)slot_of(J) * P.slot_bytes, rb, kg, p0, Re, s_xd, s_xk, x,
                                    s_part);
      }
      if (__syncthreads_or(!ok)) {
        drain_and_abort(a, bars, nslot, slot0, par0, consumed, issued, router_pend, bar_router, ph_router);
        return false;
      }
    }
    if (t + 1 == nu) split_stamp(a, l, 7);
    consumed = t * kPieces + kGuPieces;
    if ((tid & 31) == 0 && warp >= NW - kGuPieces) {
      const int j = t * kPieces + (warp - (NW - kGuPieces)) + nslot, tj = j / kPieces;
      if (j < npieces)
        issue_piece(a, W, T, NS, split_unit_of(tj, NS, s_order, a.R), j - tj * kPieces,
                    ring + (size_t)slot_of(j) * P.slot_bytes, smem_u32(bars + slot_of(j)), false);
    }
    issued = min(npieces, max(issued, t * kPieces + kGuPieces + nslot));
    // the down pieces (usually landed by now) are waited and this thread's rows loaded
    // while the SwiGLU warps work
    DnRows dr;
    {
      const int J0 = t * kPieces + kGuPieces, J1 = J0 + 1;
      split_swiglu(a, T, s_part, NG, p0, Re, s_hd);  // (warps below Re; the others go on)
      const bool ok = mbar_wait_bounded(smem_u32(bars + slot_of(J0)), par_of(J0), a.status, a.wait_cycles) &&
                      mbar_wait_bounded(smem_u32(bars + slot_of(J1)), par_of(J1), a.status, a.wait_cycles);
      if (ok) load_dn_rows(H, ring + (size_t)slot_of(J0) * P.slot_bytes, ring + (size_t)slot_of(J1) * P.slot_bytes, dr);
      if (__syncthreads_or(!ok)) {
        drain_and_abort(a, bars, nslot, slot0, par0, consumed, issued, router_pend, bar_router, ph_router);
        return false;
      }
    }
    if (t + 1 == nu) split_stamp(a, l, 8);
    split_down(a, T, dr, s_hd, p0, Re, acc_copy);
    __syncthreads();
    consumed = (t + 1) * kPieces;
    if ((tid & 31) == 0 && warp >= NW - kDnPieces) {
      const int j = t * kPieces + kGuPieces + (warp - (NW - kDnPieces)) + nslot, tj = j / kPieces;
      if (j < npieces)
        issue_piece(a, W, T, NS, split_unit_of(tj, NS, s_order, a.R), j - tj * kPieces,
                    ring + (size_t)slot_of(j) * P.slot_bytes, smem_u32(bars + slot_of(j)), false);
    }
    issued = min(npieces, max(issued, (t + 1) * kPieces + nslot));
  }
  if (nu == 0)
    for (int ph = 5; ph <= 8; ++ph) split_stamp(a, l, ph);
  return true;
}

// NG: hidden blocks in groups of 32 lanes (1 up to H 1024, 2 above).  XR: one row, its
// activation pairs in registers.  XS: the rows are staged as pairs in shared memory.
template <int NG, bool XR, bool XS>
__global__ void __launch_bounds__(NT, 1) k_split(const __grid_constant__ RoundArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5;
  const int G = gridDim.x, H = a.H, NS = a.I >> 5;
  // the plan lives in shared memory: its fields are read where they are used instead of
  // being held in registers across the layer loop
  if (tid == 0) g_splan = split_plan(a.H, a.I, a.E, a.R, a.k, G);
  __syncthreads();
  const SplitPlan& P = g_splan;
  const int nslot = P.nslot;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bars);
  const uint32_t bar_router = smem_u32(bars + nslot);
  uint8_t* ring = smem + P.ring;
  float* s_rw = reinterpret_cast<float*>(smem + P.router);
  uint4* s_xd = reinterpret_cast<uint4*>(smem + P.xd);
  uint4* s_xk = reinterpret_cast<uint4*>(smem + P.xk);
  int* s_range = reinterpret_cast<int*>(smem + P.misc);
  Tables T{reinterpret_cast<int*>(smem + P.uni),     reinterpret_cast<int*>(smem + P.csr),
           reinterpret_cast<int*>(smem + P.pair),    reinterpret_cast<float*>(smem + P.w),
           reinterpret_cast<int*>(smem + P.nunion),  reinterpret_cast<int*>(smem + P.pos_ui),
           reinterpret_cast<int*>(smem + P.pos_row), reinterpret_cast<int*>(smem + P.slot),
           reinterpret_cast<int*>(smem + P.pick)};
  unsigned* s_mask = reinterpret_cast<unsigned*>(ring);
  int* s_off_e = reinterpret_cast<int*>(ring + (size_t)a.E * 4);
  int* s_ids = reinterpret_cast<int*>(ring + (size_t)a.E * 8);
  int* s_ui = reinterpret_cast<int*>(ring + (size_t)a.E * 8 + (size_t)a.R * a.k * 4);
  int* s_rank = s_ui + a.E;
  const int o0 = (int)(((long long)blockIdx.x * H) / G);
  const int no = (int)(((long long)(blockIdx.x + 1) * H) / G) - o0;
  const int fin0 = NT / 2;  // first thread of the output finishing pass
  if (tid == 0) {
    for (int i = 0; i <= nslot; ++i) mbar_init(smem_u32(bars + i), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    issue_router_rows(a, a.layer[0].router, s_rw, bar_router);
  }
  // the accumulator copies of this CTA's output slice start at zero (ordered before any
  // other CTA's adds by the first grid barrier)
  if (!a.route_only)
    for (int i = tid; i < 2 * kSplitCopies * a.R * no; i += NT) {
      const int c = i / (a.R * no), rem = i - c * (a.R * no), r = rem / no;
      __stcg(a.acc + ((size_t)c * a.R + r) * H + o0 + (rem - r * no), 0ull);
    }
  __syncthreads();
  unsigned ph_router = 0u;
  const bool has_rows = router_rows_of_cta(a.E) > 0;
  bool router_pend = has_rows;  // layer 0's rows are in flight
  Sync sy;
  // ring position of the next layer's first piece: slot and the parity of that slot's use
  unsigned slot0 = 0u, par0 = 0u;
  for (int l = 0; l < a.L; ++l) {
    const LayerPtrs& W = a.layer[l];
    const uint16_t* x = a.x + (size_t)l * a.R * H;
    split_stamp(a, l, 0);
    if (tid == 0 && l + 1 < a.L)  // the next layer's rows into L2 (its router reads them)
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(x + (size_t)a.R * H),
                   "r"((unsigned)(a.R * H * 2))
                   : "memory");
    if (router_pend) {
      const bool ok = mbar_wait_bounded(bar_router, ph_router, a.status, a.wait_cycles);
      if (__syncthreads_or(!ok)) {
        drain_and_abort(a, bars, nslot, 0u, 0u, 0, 0, true, bar_router, ph_router);
        return;
      }
      ph_router ^= 1u;
      router_pend = false;
    }
    router_phase(a, x, s_rw);
    split_stamp(a, l, 1);
    grid_arrive(a, sy);  // B1 (all logits written)
    // the router rows are consumed: the next layer's move in
    if (tid == 0 && l + 1 < a.L) issue_router_rows(a, a.layer[l + 1].router, s_rw, bar_router);
    router_pend = has_rows && l + 1 < a.L;
    for (int e = tid; e < a.E; e += NT) {
      s_mask[e] = 0u;
      s_rank[e] = INT_MAX;
      int sl = e;
      if (W.slot) {
        sl = __ldg(W.slot + e);
        if ((unsigned)sl >= (unsigned)W.n_slots) {
          atomicOr(a.status, kStatusBadSlot);
          sl = 0;
        }
      }
      T.slot[e] = sl;
    }
    if (XS && !a.route_only) stage_xdigits(a, x, s_xd, s_xk);
    // the previous layer's output slice (upper half of the threads) while the logits
    // barrier completes: every add of that layer went into the other accumulator buffer
    // and is in (its closing barrier is behind us)
    if (l > 0 && !a.route_only) split_finish(a, l - 1, o0, no, fin0);
    if (!grid_wait(a, sy)) {
      drain_and_abort(a, bars, nslot, 0u, 0u, 0, 0, router_pend, bar_router, ph_router);
      return;
    }
    split_stamp(a, l, 2);
    const int U = route_phase(a, T, s_mask, s_off_e, s_ids, s_ui, s_rank, l, 0, NS, s_range);
    const bool one = route_one_ok(a);
    if (a.route_only) {
      if (one && warp == 1) softmax_one(a, T);
      return;
    }
    // the union's experts by row count descending, then union index (one row: all
    // weigh the same and the union's order is used as is)
    int* s_order = reinterpret_cast<int*>(smem + P.order);
    if (a.R > 1) {
      for (int ui = tid; ui < U; ui += NT) {
        const int re = T.csr_off[ui + 1] - T.csr_off[ui];
        int rank = 0;
        for (int uj = 0; uj < U; ++uj) {
          const int rj = T.csr_off[uj + 1] - T.csr_off[uj];
          rank += (rj > re || (rj == re && uj < ui)) ? 1 : 0;
        }
        s_order[rank] = ui;
      }
      __syncthreads();
    }
    split_stamp(a, l, 3);
    const int nu = split_unit_count(U * NS), npieces = nu * kPieces;
    const int n_init = min(nslot, npieces);
    // lane 0 of one warp per piece (a warp's lanes would issue their copies one after
    // another); the refills inside the unit loop likewise come from the last warps
    if ((tid & 31) == 0 && warp < n_init) {
      const int q = (int)((slot0 + (unsigned)warp) % (unsigned)nslot), tj = warp / kPieces;
      issue_piece(a, W, T, NS, split_unit_of(tj, NS, s_order, a.R), warp - tj * kPieces, ring + (size_t)q * P.slot_bytes,
                  smem_u32(bars + q));
    }
    if (one && warp == 1) softmax_one(a, T);
    split_stamp(a, l, 4);
    __syncthreads();
    if (!split_units<NG, XR, XS>(a, l, smem, slot0, par0, nu, n_init, router_pend, bar_router, ph_router))
      return;
    {
      const unsigned end = slot0 + (unsigned)npieces;
      par0 ^= (end / (unsigned)nslot) & 1u;
      slot0 = end % (unsigned)nslot;
    }
    split_stamp(a, l, 9);
    if (!grid_sync(a, sy)) {  // B3: every add of this layer is in
      drain_and_abort(a, bars, nslot, 0u, 0u, 0, 0, router_pend, bar_router, ph_router);
      return;
    }
    split_stamp(a, l, 10);
  }
  split_finish(a, a.L - 1, o0, no, fin0);
}

// ---------------------------------------------------------------------------------
// Wide verify rounds (at least kMmaRows rows): gate/up and down on the tensor cores
// (mma.sync m16n8k16, bf16 operands, fp32 accumulation), SwiGLU outputs exchanged
// between CTAs through the workspace.
//
// Per layer, with grid-wide barriers B1..B3 in between:
//   P1  router GEMV (as above)
//   B1
//   P2  routing (as above)
//   P3  gate/up: the U * I units (gate row i + up row i of a union expert) are split
//       contiguously across CTAs by work and streamed through shared-memory slots with
//       1-D bulk copies; h' = w silu(g) v goes to the workspace split into bf16 hi + lo.
//       Meanwhile this CTA's down rows of every union expert are prefetched into L2.
//   B2  (every h' written)
//   P4  down: units (expert, group of up to 16 of its positions, 16 output rows) split
//       across CTAs, on the tensor cores, the group's h' and the unit's down codes
//       staged in shared memory (two items in flight); each y * 2^32, rounded, is added
//       into the int64 accumulator of its row (exact, so order-free), and after B3 each
//       CTA sums the accumulator copies of its output slice (the next layer's B1 window).
//   B3  (layer l+1's router waits for layer l's output)
//
// A nibble n in the low four bits of a bf16 whose other bits are those of 128.0 is the
// bf16 value 128 + n, exactly; one mask-and-or per pair of weights (two nibbles 16 bits
// apart land in the two halves of a bf16x2 register), and one bf16x2 subtraction of 136
// gives n - 8, again exactly.  Inside each 32-element block the MMA's k order is
// permuted so that thread t's A fragments for the block's two k16 steps are exactly
// the eight nibbles of 32-bit word t of a row's 16-byte block:
//   step 0: k (2t, 2t+1) <- elements (8t, 8t+4),   k (2t+8, 2t+9) <- (8t+1, 8t+5)
//   step 1: k (2t, 2t+1) <- (8t+2, 8t+6),          k (2t+8, 2t+9) <- (8t+3, 8t+7)
// The B fragments (activations, or the exchanged h' split into bf16 hi + lo) follow the
// same permutation.  A block's MMAs give sum (n - 8) b, which the block scale then
// multiplies into the fp32 accumulator.  Each warp keeps one A tile (16 weight rows x
// one K part) in registers for up to two n-tiles (16 expert rows or positions).  Every
// tile's K range is split in the same fixed parts whatever the other rows are, and the
// parts are added in a fixed order, so a row's result does not depend on the rows it
// shares the round with.

// Rounds of at least this many rows use the tensor-core kernel.  The choice is made
// before the routing is known.  Measured on the 128-expert / top-8 layer (40-layer
// rounds): with 14 to 16 near-duplicate copy-span rows (about 11 experts per layer) the
// tensor cores take 39 to 40 us per layer against 65 to 72 us on the split kernel; with
// draft rows at sigma 0.5 (about 27 experts) the split kernel is faster from 13 rows on
// (56 against 65 us at 13 rows, 65 against 69 us at 16) and below 13 rows for every row
// mix measured.  The switch favours the copy-span rounds.
constexpr int kMmaRows = 13;
constexpr int kKPartsGu = 8;  // K parts of a gate/up tile (hidden blocks)
static_assert(NW % kKPartsGu == 0, "a tile's K parts run in one round");
constexpr int kGuSlots = 3;
// scratch of the tensor-core path
constexpr int kMmaMaxPos = 256;          // CSR positions (rows x top-k) of a wide round
constexpr size_t kMmaPart = 0;           // [NW][2][16][8] fp32 partial tiles
constexpr size_t kMmaScratch = (size_t)NW * 256 * 4;

// Intermediate blocks of one staged down item: the largest of 24, 16, 8 dividing I / 32.
__host__ __device__ inline int dn_item_blocks(int NBI) { return NBI % 24 == 0 ? 24 : (NBI % 16 == 0 ? 16 : 8); }
// The down pass's staging: one h' chunk [16 positions][KB blocks][128 B] and a ring of
// kDnRing unit slots, each the unit's codes [KB][16 rows][16 B] and scales [KB][16 fp16].
constexpr int kDnRing = 16;  // two rounds of NW / 2 units
__host__ __device__ inline size_t dn_h_bytes(int KB) { return (size_t)16 * KB * 128; }
__host__ __device__ inline size_t dn_c_bytes(int KB) { return (size_t)KB * 256; }
__host__ __device__ inline size_t dn_slot_bytes(int NBI) {
  const int KB = dn_item_blocks(NBI);
  return dn_c_bytes(KB) + (size_t)KB * 32;  // (a multiple of 16 bytes)
}
__host__ __device__ inline size_t dn_stage_bytes(int NBI) {
  return dn_h_bytes(dn_item_blocks(NBI)) + (size_t)kDnRing * dn_slot_bytes(NBI);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

struct GuChunk {
  int ui, i0, n;
};

// smem plan of the wide kernel: GU ring | MMA scratch | tables | chunk list | barriers
struct WidePlan {
  size_t gu_slot, gu, scratch, uni, csr, pair, w, pos_ui, pos_row, slot, pick, nunion, chunks, bars, total;
  size_t ring;
  size_t dn, dn_slot;  // the down pass's staging: offset in the ring, bytes of one unit slot
  int gu_cap;     // units per gate/up chunk
  bool ok;
};

__host__ __device__ inline WidePlan wide_plan(int H, int I, int E, int R, int k, int grid) {
  WidePlan p{};
  const size_t unit = (size_t)H + (size_t)H / 8;
  const size_t tables = up128((size_t)E * 4) + up128((size_t)(E + 1) * 4) + 5 * up128((size_t)R * k * 4) +
                        up128((size_t)E * 4) + 128 + up128(kGuSlots * 12 + 64) + 256;
  const size_t fixed = tables + kMmaScratch;
  const size_t limit = (size_t)225 * 1024;
  size_t cap = fixed < limit ? ((limit - fixed) / kGuSlots) / unit : 0;
  if (cap > NW) cap = NW;  // a chunk is one pass of the warps
  p.gu_cap = (int)cap;
  p.gu_slot = up128(cap * unit);
  const int rows_per_cta = (E + grid - 1) / grid;
  p.ring = kGuSlots * p.gu_slot;
  const size_t scratch_need = ((size_t)4 * E + (size_t)R * k) * 4 + 16 + (size_t)(5 * NT + NW) * 4;
  const size_t router_need = (size_t)rows_per_cta * H * 4;
  if (p.ring < scratch_need) p.ring = up128(scratch_need);
  if (p.ring < router_need) p.ring = up128(router_need);
  // the down pass stages through the ring past the next layer's router rows
  p.dn = up128(router_need);
  p.dn_slot = dn_slot_bytes(I >> 5);
  if (p.ring < p.dn + dn_stage_bytes(I >> 5)) p.ring = up128(p.dn + dn_stage_bytes(I >> 5));

  size_t off = 0;
  p.gu = off;      off += p.ring;
  p.scratch = off; off += kMmaScratch;
  p.uni = off;     off += up128((size_t)E * 4);
  p.csr = off;     off += up128((size_t)(E + 1) * 4);
  p.pair = off;    off += up128((size_t)R * k * 4);
  p.w = off;       off += up128((size_t)R * k * 4);
  p.pos_ui = off;  off += up128((size_t)R * k * 4);
  p.pos_row = off; off += up128((size_t)R * k * 4);
  p.slot = off;    off += up128((size_t)E * 4);
  p.pick = off;    off += up128((size_t)R * k * 4);
  p.nunion = off;  off += 128;
  p.chunks = off;  off += up128(kGuSlots * 12 + 64);
  p.bars = off;    off += 256;
  p.total = off;
  p.ok = cap >= 8 && (size_t)R * k <= kMmaMaxPos && p.total <= limit;
  return p;
}

__device__ void issue_gu_chunk(const RoundArgs& a, const LayerPtrs& W, const Tables& T, uint8_t* dst,
                               uint32_t bar, const GuChunk& c) {
  const size_t H = (size_t)a.H, I = (size_t)a.I;
  const size_t u = (size_t)T.slot[T.uni[c.ui]];
  const size_t first = u * I + (size_t)c.i0;  // unit index within the bank
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_expect_tx(bar, (uint32_t)((size_t)c.n * (H + H / 8)));
  bulk_g2s(smem_u32(dst), W.gu_nib + first * H, (uint32_t)(c.n * H), bar);
  bulk_g2s(smem_u32(dst + (size_t)c.n * H),
           reinterpret_cast<const uint8_t*>(W.gu_sc) + first * (H / 8), (uint32_t)(c.n * (H / 8)), bar);
}

// Gate/up of one staged chunk on the tensor cores.  A tile = 8 units of the chunk (A
// row g: the gate row of unit g, row g + 8: its up row, so the eight lanes' rows have
// eight different block swizzles) x up to 16 of the expert's rows (two n-tiles) x one
// of kKPartsGu K parts; one warp per tile part.  The parts are added in order, then
// h' = w silu(g) v is stored split into bf16 hi + lo in the down pass's fragment order.
__device__ void gateup_chunk_mma(const RoundArgs& a, const Tables& T, const uint8_t* slot, const GuChunk& c,
                                 const uint16_t* x, float* s_part) {
  const int H = a.H, NB = H >> 5, NBI = a.I >> 5;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int p0 = T.csr_off[c.ui], Re = T.csr_off[c.ui + 1] - p0;
  const int NTP = (Re + 15) >> 4, MT = (c.n + 7) >> 3, n_asg = MT * NTP * kKPartsGu;
  const uint8_t* codes = slot;
  const uint16_t* scales = reinterpret_cast<const uint16_t*>(slot + (size_t)c.n * H);
  uint16_t* hb = reinterpret_cast<uint16_t*>(a.hbuf);
  for (int j0 = 0; j0 < n_asg; j0 += NW) {
    const int j = j0 + warp;
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if (j < n_asg) {
      const int gi = j / kKPartsGu, kp = j - gi * kKPartsGu;
      const int mt = gi / NTP, ntp = gi - mt * NTP;
      // units past the chunk repeat its last one; their results are dropped
      const int u = min(mt * 8 + g, c.n - 1), kk = (c.i0 + u) & 7;
      const uint32_t* wg = reinterpret_cast<const uint32_t*>(codes + (size_t)(2 * u) * NB * 16) + t;
      const uint32_t* wu = wg + NB * 4;
      const uint16_t* sg_ = scales + (size_t)(2 * u) * NB;
      const uint16_t* su_ = sg_ + NB;
      // columns past the expert's rows repeat its last row; their results are dropped
      const int c0 = ntp * 16 + g;
      const bool two = ntp * 16 + 8 < Re;
      const uint4* x0 = reinterpret_cast<const uint4*>(x + (size_t)T.pos_row[p0 + min(c0, Re - 1)] * H) + t;
      const uint4* x1 = reinterpret_cast<const uint4*>(x + (size_t)T.pos_row[p0 + min(c0 + 8, Re - 1)] * H) + t;
      const int b0 = (kp * NB) / kKPartsGu, b1 = ((kp + 1) * NB) / kKPartsGu;
#pragma unroll 2
      for (int b = b0; b < b1; ++b) {
        const int pb = b ^ kk;
        uint32_t pg[4], pu[4];
        dq_word(wg[4 * pb], pg);
        dq_word(wu[4 * pb], pu);
        const float sg = half_bits(sg_[pb]), su = half_bits(su_[pb]);
        {
          uint32_t bf[4];
          bfrag_x(__ldg(x0 + 4 * b), bf);
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          mma_bf16(d, pg[0], pu[0], pg[1], pu[1], bf[0], bf[1]);
          mma_bf16(d, pg[2], pu[2], pg[3], pu[3], bf[2], bf[3]);
          acc[0][0] = __fmaf_rn(sg, d[0], acc[0][0]);
          acc[0][1] = __fmaf_rn(sg, d[1], acc[0][1]);
          acc[0][2] = __fmaf_rn(su, d[2], acc[0][2]);
          acc[0][3] = __fmaf_rn(su, d[3], acc[0][3]);
        }
        if (two) {
          uint32_t bf[4];
          bfrag_x(__ldg(x1 + 4 * b), bf);
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          mma_bf16(d, pg[0], pu[0], pg[1], pu[1], bf[0], bf[1]);
          mma_bf16(d, pg[2], pu[2], pg[3], pu[3], bf[2], bf[3]);
          acc[1][0] = __fmaf_rn(sg, d[0], acc[1][0]);
          acc[1][1] = __fmaf_rn(sg, d[1], acc[1][1]);
          acc[1][2] = __fmaf_rn(su, d[2], acc[1][2]);
          acc[1][3] = __fmaf_rn(su, d[3], acc[1][3]);
        }
      }
    }
    store_part(s_part + warp * 256, acc, g, t);
    __syncthreads();
    for (int i = threadIdx.x; i < (NW / kKPartsGu) * 128; i += NT) {
      const int gl = i >> 7, nt = (i >> 6) & 1, uu = (i >> 3) & 7, cc = i & 7;
      const int gi = j0 / kKPartsGu + gl;
      if (gi >= MT * NTP) continue;
      const int mt = gi / NTP, ntp = gi - mt * NTP;
      const int u = mt * 8 + uu, col = ntp * 16 + nt * 8 + cc;
      if (u >= c.n || col >= Re) continue;
      float gs = 0.f, vs = 0.f;
#pragma unroll
      for (int kp = 0; kp < kKPartsGu; ++kp) {
        const float* Pp = s_part + (gl * kKPartsGu + kp) * 256 + nt * 128;
        gs = __fadd_rn(gs, Pp[uu * 8 + cc]);
        vs = __fadd_rn(vs, Pp[64 + uu * 8 + cc]);
      }
      const int pp = p0 + col;
      const float hh = __fmul_rn(__fdiv_rn(gs, __fadd_rn(1.f, expf(-gs))), vs);
      const float hw = __fmul_rn(T.w[T.pair[pp]], hh);
      const __nv_bfloat16 hi = __float2bfloat16_rn(hw);
      const __nv_bfloat16 lo = __float2bfloat16_rn(__fsub_rn(hw, __bfloat162float(hi)));
      const int i2 = c.i0 + u, jj = i2 & 31, e = jj & 7;
      const size_t base = (((size_t)pp * NBI + (i2 >> 5)) * 4 + (jj >> 3)) * 16 + 2 * (e & 3) + (e >> 2);
      hb[base] = __bfloat16_as_ushort(hi);
      hb[base + 8] = __bfloat16_as_ushort(lo);
    }
    __syncthreads();
  }
}

// The down units [du0, du1) of this CTA (unit = (expert group, block of 16 output rows),
// as the down pass numbers them) into L2: they depend only on the routing and are read
// after the h exchange.  Per unit and intermediate block, one bulk prefetch of the 16
// rows' codes (256 bytes) and one of their scales (32 bytes).
__device__ void prefetch_down_units(const RoundArgs& a, const LayerPtrs& W, const Tables& T, int gpe, int du0,
                                    int du1) {
  const int NBI = a.I >> 5, H = a.H, NOB = H >> 4;
  for (int i = threadIdx.x; i < (du1 - du0) * NBI; i += NT) {
    const int du = du0 + i / NBI, b = i - (i / NBI) * NBI;
    const int ug = du / NOB, ob = du - ug * NOB, ui = ug / gpe;
    if (16 * (ug - ui * gpe) >= T.csr_off[ui + 1] - T.csr_off[ui]) continue;  // an empty group
    const size_t row = ((size_t)T.slot[T.uni[ui]] * NBI + b) * H + (size_t)ob * 16;
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(W.dn_nib + row * 16), "r"(256u) : "memory");
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(W.dn_sc + row), "r"(32u) : "memory");
  }
}

__global__ void __launch_bounds__(NT, 1) k_round(const __grid_constant__ RoundArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  const int tid = threadIdx.x;
  const int G = gridDim.x;
  const WidePlan P = wide_plan(a.H, a.I, a.E, a.R, a.k, G);
  // mbarriers: kGuSlots GU slots, the router rows
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bars);
  const uint32_t bar_router = smem_u32(bars + kGuSlots);
  uint8_t* gu = smem + P.gu;
  float* s_mpart = reinterpret_cast<float*>(smem + P.scratch + kMmaPart);
  float* s_rw = reinterpret_cast<float*>(gu);
  GuChunk* s_chunks = reinterpret_cast<GuChunk*>(smem + P.chunks);
  Tables T{reinterpret_cast<int*>(smem + P.uni),     reinterpret_cast<int*>(smem + P.csr),
           reinterpret_cast<int*>(smem + P.pair),    reinterpret_cast<float*>(smem + P.w),
           reinterpret_cast<int*>(smem + P.nunion),  reinterpret_cast<int*>(smem + P.pos_ui),
           reinterpret_cast<int*>(smem + P.pos_row), reinterpret_cast<int*>(smem + P.slot),
           reinterpret_cast<int*>(smem + P.pick)};
  // routing scratch lives in the (then idle) gate/up ring
  unsigned* s_mask = reinterpret_cast<unsigned*>(gu);
  int* s_off_e = reinterpret_cast<int*>(gu + (size_t)a.E * 4);
  int* s_ids = reinterpret_cast<int*>(gu + (size_t)a.E * 8);
  int* s_ui = reinterpret_cast<int*>(gu + (size_t)a.E * 8 + (size_t)a.R * a.k * 4);
  int* s_rank = s_ui + a.E;
  if (tid == 0) {
    for (int i = 0; i < kGuSlots + 2; ++i) mbar_init(smem_u32(bars + i), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    issue_router_rows(a, a.layer[0].router, s_rw, bar_router);
  }
  __syncthreads();
  unsigned ph_router = 0u;
  bool router_pend = router_rows_of_cta(a.E) > 0;  // layer 0's rows are in flight
  Sync sy;
  unsigned gu_ph = 0u;            // bit q: parity of GU slot q
  const size_t RH = (size_t)a.R * a.H;
  const int o0 = (int)(((long long)blockIdx.x * a.H) / G);
  const int no = (int)(((long long)(blockIdx.x + 1) * a.H) / G) - o0;
  // this CTA's output slice of the accumulators (one copy per layer parity: an output
  // receives only its row's k adds here) starts at zero, ordered before any other CTA's
  // adds by the first grid barrier
  for (int i = tid; i < 2 * a.R * no; i += NT) {
    const int c = i / (a.R * no), rem = i - c * (a.R * no), r = rem / no;
    __stcg(a.acc + ((size_t)c * kAccCopies * a.R + r) * a.H + o0 + (rem - r * no), 0ull);
  }
  // the GU slots in flight: bit q set
  unsigned gu_pend = 0u;
  // the down pass's h' chunk (thread 0's view): parity of its next completion, in flight
  const uint32_t bar_dn = smem_u32(bars + kGuSlots + 1);
  unsigned dn_ph = 0u, dn_pend = 0u;
  auto bail = [&]() {
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (tid == 0) {
      for (int q = 0; q < kGuSlots; ++q)
        if (gu_pend & (1u << q)) mbar_wait_bounded(smem_u32(bars + q), (gu_ph >> q) & 1u, a.status, kDefaultWaitCycles);
      if (dn_pend) mbar_wait_bounded(bar_dn, dn_ph, a.status, kDefaultWaitCycles);
    }
    drain_and_abort(a, bars, 1, 0u, 0u, 0, 0, router_pend, bar_router, ph_router);
  };
  for (int l = 0; l < a.L; ++l) {
    const LayerPtrs& W = a.layer[l];
    const uint16_t* x = a.x + (size_t)l * RH;
    stamp(a, l, 0);
    if (router_pend) {
      const bool ok = mbar_wait_bounded(bar_router, ph_router, a.status, a.wait_cycles);
      if (__syncthreads_or(!ok)) {
        bail();
        return;
      }
      ph_router ^= 1u;
      router_pend = false;
    }
    router_phase(a, x, s_rw);
    stamp(a, l, 1);
    grid_arrive(a, sy);  // B1 (all logits written)
    for (int e = tid; e < a.E; e += NT) {  // (the router rows there are consumed)
      s_mask[e] = 0u;
      s_rank[e] = INT_MAX;
      int sl = e;
      if (W.slot) {
        sl = __ldg(W.slot + e);
        if ((unsigned)sl >= (unsigned)W.n_slots) {
          atomicOr(a.status, kStatusBadSlot);
          sl = 0;
        }
      }
      T.slot[e] = sl;
    }
    // the previous layer's output slice while the logits barrier completes (every add of
    // that layer went into the other accumulator buffer and is in: its closing barrier is
    // behind us)
    if (l > 0 && no > 0) split_finish(a, l - 1, o0, no, 0, 1);
    if (!grid_wait(a, sy)) {
      bail();
      return;
    }
    stamp(a, l, 2);
    int* s_range = reinterpret_cast<int*>(smem + P.chunks + kGuSlots * 12 + 20);
    const int U = route_phase(a, T, s_mask, s_off_e, s_ids, s_ui, s_rank, l, 1, a.I, s_range);
    stamp(a, l, 3);
    // ---- this CTA's share of the gate/up units (cut during routing); chunks issued
    // through the ring: thread 0 cuts them lazily (stopping at expert boundaries and the
    // slot size) and leaves the descriptor of chunk n in ring entry n % kGuSlots ----
    int* s_cursor = reinterpret_cast<int*>(smem + P.chunks + kGuSlots * 12 + 4);
    auto next_chunk = [&](int cap) {
      int cur = s_cursor[0], ui = s_cursor[2], i0 = s_cursor[3];
      int nn = s_cursor[1] - cur;
      if (nn > a.I - i0) nn = a.I - i0;
      if (nn > cap) nn = cap;
      const GuChunk ch{ui, i0, nn};
      cur += nn;
      i0 += nn;
      if (i0 == a.I) {
        ++ui;
        i0 = 0;
      }
      s_cursor[0] = cur;
      s_cursor[2] = ui;
      s_cursor[3] = i0;
      return ch;
    };
    const int g_cur = s_range[0], g_end = s_range[1];
    if (tid == 0) {
      s_cursor[0] = g_cur;
      s_cursor[1] = g_end;
      s_cursor[2] = g_cur / a.I;
      s_cursor[3] = g_cur - (g_cur / a.I) * a.I;
      int nc = 0;
      for (int cur = g_cur, i0 = s_cursor[3]; cur < g_end; ++nc) {
        int nn = g_end - cur;
        if (nn > a.I - i0) nn = a.I - i0;
        if (nn > P.gu_cap) nn = P.gu_cap;
        cur += nn;
        i0 = (i0 + nn == a.I) ? 0 : i0 + nn;
      }
      for (int q = 0; q < kGuSlots && q < nc; ++q) {
        s_chunks[q] = next_chunk(P.gu_cap);
        issue_gu_chunk(a, W, T, gu + q * P.gu_slot, smem_u32(bars + q), s_chunks[q]);
      }
      *reinterpret_cast<int*>(smem + P.chunks + kGuSlots * 12) = nc;
    }
    // this CTA's down units are needed after B2: into L2 now
    {
      const int gpe = (a.R + 15) >> 4;
      const unsigned n_du = (unsigned)U * (unsigned)gpe * (unsigned)(a.H >> 4);
      prefetch_down_units(a, W, T, gpe, (int)(((unsigned)blockIdx.x * n_du) / (unsigned)G),
                          (int)((((unsigned)blockIdx.x + 1u) * n_du) / (unsigned)G));
    }
    __syncthreads();
    const int n_chunks = *reinterpret_cast<const int*>(smem + P.chunks + kGuSlots * 12);
    gu_pend = (1u << min(kGuSlots, n_chunks)) - 1u;
    // ---- gate/up ----
    for (int n = 0; n < n_chunks; ++n) {
      const int q = n % kGuSlots;
      const bool ok = mbar_wait_bounded(smem_u32(bars + q), (gu_ph >> q) & 1u, a.status, a.wait_cycles);
      if (__syncthreads_or(!ok)) {
        bail();
        return;
      }
      gu_ph ^= 1u << q;
      gu_pend &= ~(1u << q);
      if (n == 0) stamp(a, l, 4);
      stamp(a, l, 5);  // (the last chunk's stamp stays)
      const GuChunk c = s_chunks[q];
      gateup_chunk_mma(a, T, gu + q * P.gu_slot, c, x, s_mpart);
      __syncthreads();  // slot q free again
      if (n + kGuSlots < n_chunks) {
        gu_pend |= 1u << q;
        if (tid == 0) {
          s_chunks[q] = next_chunk(P.gu_cap);
          issue_gu_chunk(a, W, T, gu + q * P.gu_slot, smem_u32(bars + q), s_chunks[q]);
        }
      }
    }
    if (n_chunks == 0) {
      stamp(a, l, 4);
      stamp(a, l, 5);
    }
    // the next layer's router rows can move in now (the GU ring is idle until then)
    if (l + 1 < a.L && router_rows_of_cta(a.E) > 0) {
      router_pend = true;
      if (tid == 0) issue_router_rows(a, a.layer[l + 1].router, s_rw, bar_router);
    }
    stamp(a, l, 6);
    if (!grid_sync(a, sy)) {  // B2: every h written
      bail();
      return;
    }
    stamp(a, l, 7);
    stamp(a, l, 8);
    {
      // ---- wide down on the tensor cores ----
      // Units (union expert, group of up to 16 of its positions, block of 16 output rows),
      // in that order, split contiguously across the CTAs: a CTA's units share one or two
      // groups, and each expert's h' is read by the few CTAs that own its rows (a pass
      // sliced by output rows makes every CTA read every expert's h').  Per group segment
      // of the range and K chunk of KB blocks, the group's h' chunk is staged once (bulk
      // copy); the units' codes and scales stream through a ring of kDnRing slots by
      // cp.async, in rounds of NW / 2 units.  Warp = (unit of the round, n-tile) over the
      // whole chunk: two MMAs per k16 step (h' hi + lo), the block scale applied per block,
      // and each y[position][row] * 2^32, rounded, is added into the int64 accumulator of
      // the position's row (exact integer adds: the output depends on neither the order,
      // the split nor the other rows).
      const int gpe = (a.R + 15) >> 4;  // position groups per expert
      const int H = a.H, NOB = H >> 4, NBI = a.I >> 5, KB = dn_item_blocks(NBI), NKC = NBI / KB;
      const unsigned n_du = (unsigned)U * (unsigned)gpe * (unsigned)NOB;
      const int du0 = (int)(((unsigned)blockIdx.x * n_du) / (unsigned)G);
      const int du1 = (int)((((unsigned)blockIdx.x + 1u) * n_du) / (unsigned)G);
      const uint8_t* hb = reinterpret_cast<const uint8_t*>(a.hbuf);
      unsigned long long* acc_copy = a.acc + (size_t)(l & 1) * kAccCopies * RH;
      uint8_t* sh = gu + P.dn;                 // the h' chunk
      uint8_t* ring_dn = sh + dn_h_bytes(KB);  // unit slots
      constexpr int kRound = NW / 2;
      const int lane = tid & 31, g = lane >> 2, t = lane & 3, wq = (tid >> 5) >> 1, nt = (tid >> 5) & 1;
      if (du0 < du1 && tid == 0)  // h' was written by generic stores before B2; bulk copies read it
        asm volatile("fence.proxy.async.global;" ::: "memory");
      for (int sg = du0; sg < du1;) {
        const int ug = sg / NOB, ob0 = sg - ug * NOB;
        const int seg_end = min(du1, (ug + 1) * NOB), nu = seg_end - sg;
        const int ui = ug / gpe, p0 = T.csr_off[ui] + 16 * (ug - ui * gpe);
        const int cnt = min(16, T.csr_off[ui + 1] - p0);
        sg = seg_end;
        if (cnt <= 0) continue;  // an empty group (uniform)
        const size_t blk0 = (size_t)T.slot[T.uni[ui]] * NBI;
        const int nr = (nu + kRound - 1) / kRound;
        for (int kc = 0; kc < NKC; ++kc) {
          // the group's h' chunk (its previous readers are past the last barrier)
          if (tid == 0) {
            const uint32_t bytes = (uint32_t)(cnt * KB * 128);
            mbar_expect_tx(bar_dn, bytes);
            if (NKC == 1) {
              bulk_g2s(smem_u32(sh), hb + (size_t)p0 * NBI * 128, bytes, bar_dn);
            } else {
              for (int q = 0; q < cnt; ++q)
                bulk_g2s(smem_u32(sh + (size_t)q * KB * 128), hb + ((size_t)(p0 + q) * NBI + (size_t)kc * KB) * 128,
                         (uint32_t)(KB * 128), bar_dn);
            }
            dn_pend = 1u;
          }
          // round r: units kRound r .. of the segment, unit j in ring slot j % kDnRing: codes
          // (block b of the 16 rows is one 256-byte run) and scales (32 bytes per block)
          auto issue_round = [&](int r) {
            const int j0 = r * kRound, nj = min(kRound, nu - j0);
            for (int i = tid; i < nj * KB * 18; i += NT) {
              const int q = i / (KB * 18), e = i - q * (KB * 18), j = j0 + q;
              uint8_t* sc = ring_dn + (size_t)(j % kDnRing) * P.dn_slot;
              const size_t row0 = (blk0 + (size_t)kc * KB) * (size_t)H + (size_t)(ob0 + j) * 16;
              if (e < KB * 16)
                cp_async16(smem_u32(sc + (size_t)e * 16), W.dn_nib + (row0 + (size_t)(e >> 4) * H + (e & 15)) * 16);
              else {
                const int f = e - KB * 16;  // scales: block f / 2, half f & 1 of its 16 values
                cp_async16(smem_u32(sc + dn_c_bytes(KB) + (size_t)f * 16),
                           W.dn_sc + row0 + (size_t)(f >> 1) * H + (f & 1) * 8);
              }
            }
            cp_async_commit();
          };
          issue_round(0);
          if (nr > 1) issue_round(1);
          // (every thread waits: the wait is its acquire of the copied bytes)
          const bool ok = mbar_wait_bounded(bar_dn, dn_ph, a.status, a.wait_cycles);
          if (ok) {
            dn_ph ^= 1u;
            dn_pend = 0u;
          }
          // positions past the group repeat its last one; their results are dropped
          const uint4* hrow = reinterpret_cast<const uint4*>(sh + (size_t)min(nt * 8 + g, cnt - 1) * KB * 128) + 2 * t;
          for (int r = 0; r < nr; ++r) {
            if (r + 1 < nr)
              cp_async_wait<1>();
            else
              cp_async_wait<0>();
            if (__syncthreads_or(!ok)) {
              bail();
              return;
            }
            const int j = r * kRound + wq;
            if (j < nu && nt * 8 < cnt) {
              const uint8_t* sc = ring_dn + (size_t)(j % kDnRing) * P.dn_slot;
              const uint16_t* s16 = reinterpret_cast<const uint16_t*>(sc + dn_c_bytes(KB));
              const uint32_t* ca = reinterpret_cast<const uint32_t*>(sc) + g * 4 + t;
              float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
              for (int b = 0; b < KB; ++b) {
                uint32_t fa[4], fb[4];
                dq_word(ca[b * 64], fa);
                dq_word(ca[b * 64 + 32], fb);
                const float sa = half_bits(s16[b * 16 + g]), sbb = half_bits(s16[b * 16 + g + 8]);
                const uint4 hi = hrow[8 * b], lo = hrow[8 * b + 1];
                float d[4] = {0.f, 0.f, 0.f, 0.f};
                mma_bf16(d, fa[0], fb[0], fa[1], fb[1], hi.x, hi.y);
                mma_bf16(d, fa[0], fb[0], fa[1], fb[1], lo.x, lo.y);
                mma_bf16(d, fa[2], fb[2], fa[3], fb[3], hi.z, hi.w);
                mma_bf16(d, fa[2], fb[2], fa[3], fb[3], lo.z, lo.w);
                acc[0] = __fmaf_rn(sa, d[0], acc[0]);
                acc[1] = __fmaf_rn(sa, d[1], acc[1]);
                acc[2] = __fmaf_rn(sbb, d[2], acc[2]);
                acc[3] = __fmaf_rn(sbb, d[3], acc[3]);
              }
              const int o = (ob0 + j) * 16 + g;
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                const int pos = nt * 8 + 2 * t + (v & 1);
                if (pos < cnt)
                  red_add_u64(acc_copy + (size_t)T.pos_row[p0 + pos] * H + o + (v >> 1) * 8,
                              (unsigned long long)__float2ll_rn(acc[v] * 4294967296.0f));
              }
            }
            __syncthreads();  // this round's slots are free
            if (r + 2 < nr) issue_round(r + 2);
          }
        }
      }
    }
    stamp(a, l, 9);
    stamp(a, l, 10);
    stamp(a, l, 11);
    if (!grid_sync(a, sy)) {  // B3: every add of this layer is in
      bail();
      return;
    }
    stamp(a, l, 12);
  }
  if (no > 0) split_finish(a, a.L - 1, o0, no, 0, 1);
}

}  // namespace
}  // namespace moe

// =====================================================================================
// host side

using namespace moe;

struct GraphKey {
  std::vector<moe_layer_w> layers;
  int32_t rows = 0;
  int32_t tail_rank = 0;
  const void *x = nullptr, *out = nullptr, *stats = nullptr, *ws = nullptr, *stream = nullptr;
  size_t ws_bytes = 0;
  bool operator==(const GraphKey& o) const {
    if (rows != o.rows || tail_rank != o.tail_rank || x != o.x || out != o.out || stats != o.stats ||
        ws != o.ws ||
        stream != o.stream || ws_bytes != o.ws_bytes || layers.size() != o.layers.size())
      return false;
    return layers.empty() ||
           std::memcmp(layers.data(), o.layers.data(), layers.size() * sizeof(moe_layer_w)) == 0;
  }
};

struct moe_handle {
  moe_dims dims;
  int device = 0;
  int sm_count = 0;
  unsigned* status = nullptr;
  unsigned long long wait_ns = kDefaultWaitNs;
  int32_t tail_rank = 0;
  int32_t last_launches = 0;
  GraphKey gkey;
  cudaGraphExec_t gexec = nullptr;
  int32_t graph_launches = 0;
  // profiling of eager calls (moe_profile): event pairs and phase stamps
  bool profiling = false;
  std::vector<cudaEvent_t> ev;  // start/stop pairs
  size_t ev_used = 0;
  long long* phase_ts = nullptr;  // [kMaxLayers][kPhases][sm_count]
  int32_t phase_layers = 0;
  int last_kind = 0;   // kernel of the most recent launch (kKindSplit / kKindWide)
  int phase_kind = 0;  // kernel of the last profiled round
};

namespace {

struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) {
      ok = false;
      prev = -1;
      return;
    }
    if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_layer(const moe_layer_w* w) {
  if (!w) return MOE_EINVAL;
  if (!aligned16(w->router) || !aligned16(w->gateup_nib) || !aligned16(w->gateup_scale) ||
      !aligned16(w->down_nib) || !aligned16(w->down_scale))
    return MOE_EINVAL;
  if (w->slot_of_expert && (w->n_slots < 1 || (reinterpret_cast<uintptr_t>(w->slot_of_expert) & 3u)))
    return MOE_EINVAL;
  return MOE_OK;
}

typedef void (*KernelFn)(RoundArgs);
enum { kKindSplit = 0, kKindWide = 1 };

// The kernel instantiations that can serve a hidden size: the split kernel with one row
// in registers, with staged rows, with rows read from global memory; the wide kernel.
struct KernelSet {
  KernelFn split_xr, split_xs, split_gx, wide;
};

KernelSet kernels_for(int H) {
  if ((((H >> 5) + 31) >> 5) == 1)
    return {k_split<1, true, true>, k_split<1, false, true>, k_split<1, false, false>, k_round};
  return {k_split<2, true, true>, k_split<2, false, true>, k_split<2, false, false>, k_round};
}

struct Choice {
  KernelFn fn = nullptr;
  size_t smem = 0;
  int kind = kKindSplit;
};

// The kernel of a call with `rows` rows: the tensor cores for rounds of at least
// kMmaRows rows whose plan fits, the split kernel otherwise.  False if neither fits.
bool choose_kernel(const moe_dims& d, int rows, int grid, bool route_only, Choice& c) {
  const KernelSet ks = kernels_for(d.hidden);
  if (!route_only && rows >= kMmaRows) {
    const WidePlan w = wide_plan(d.hidden, d.inter, d.n_experts, rows, d.top_k, grid);
    if (w.ok) {
      c.fn = ks.wide;
      c.smem = w.total;
      c.kind = kKindWide;
      return true;
    }
  }
  const SplitPlan sp = split_plan(d.hidden, d.inter, d.n_experts, rows, d.top_k, grid);
  if (!sp.ok) return false;
  c.fn = (rows == 1 && sp.x_staged) ? ks.split_xr : (sp.x_staged ? ks.split_xs : ks.split_gx);
  c.smem = sp.total;
  c.kind = kKindSplit;
  return true;
}

// The dynamic shared-memory limit is an attribute of the kernel function, shared by
// every handle: raise it once to the device's opt-in maximum (minus the kernel's static
// shared memory), so a handle created later with a smaller plan cannot lower it below
// what an earlier handle launches with.
cudaError_t allow_max_dynamic_smem(int device, KernelFn fn) {
  int optin = 0;
  cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, device);
  cudaFuncAttributes fa{};
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, fn);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
  return e;
}

// Raises the limits of every kernel that can serve hidden size H.
cudaError_t prepare_kernels(int device, int H) {
  const KernelSet ks = kernels_for(H);
  cudaError_t e = allow_max_dynamic_smem(device, ks.split_xr);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(device, ks.split_xs);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(device, ks.split_gx);
  if (e == cudaSuccess) e = allow_max_dynamic_smem(device, ks.wide);
  return e;
}

// Every row count 1..max_rows (and routing alone) has a kernel whose plan fits and of
// which one CTA fits an SM.  MOE_EUNSUPPORTED if not, MOE_ECUDA on a runtime error.
int check_plans(const moe_dims& d, int grid) {
  if ((size_t)((d.n_experts + grid - 1) / grid) * d.hidden * 4 > (size_t)64 * 1024) return MOE_EUNSUPPORTED;
  for (int rows = 1; rows <= d.max_rows; ++rows)
    for (int ro = 0; ro < 2; ++ro) {
      Choice c;
      if (!choose_kernel(d, rows, grid, ro != 0, c)) return MOE_EUNSUPPORTED;
      int occ = 0;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, c.fn, NT, c.smem) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ECUDA;
      }
      if (occ < 1) return MOE_EUNSUPPORTED;
    }
  return MOE_OK;
}

void fill_args(RoundArgs& a, const moe_handle* h, int rows, void* ws) {
  const moe_dims& d = h->dims;
  const WsLayout L = ws_layout(d, rows);
  char* base = static_cast<char*>(ws);
  a.H = d.hidden;
  a.E = d.n_experts;
  a.k = d.top_k;
  a.I = d.inter;
  a.R = rows;
  a.Rmax = d.max_rows;
  a.bar = reinterpret_cast<unsigned*>(base + L.ctrl);
  a.logits = reinterpret_cast<float*>(base + L.logits);
  a.hbuf = reinterpret_cast<float*>(base + L.hbuf);
  a.acc = reinterpret_cast<unsigned long long*>(base + L.acc);
  a.status = h->status;
  a.tail_rank = h->tail_rank;
  const unsigned long long ns = h->wait_ns < (1ull << 40) ? h->wait_ns : (1ull << 40);
  a.wait_cycles = (long long)ns * kCyclesPerNs;
}

cudaError_t launch_round(moe_handle* h, const RoundArgs& a, cudaStream_t st, bool capturing) {
  cudaError_t e = cudaMemsetAsync(a.bar, 0, 256, st);
  if (e != cudaSuccess) return e;
  const bool prof = h->profiling && !capturing;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (prof) {
    while (h->ev.size() < h->ev_used + 2) {
      cudaEvent_t ev;
      if (cudaEventCreate(&ev) != cudaSuccess) return cudaGetLastError();
      h->ev.push_back(ev);
    }
    e0 = h->ev[h->ev_used];
    e1 = h->ev[h->ev_used + 1];
    h->ev_used += 2;
    cudaEventRecord(e0, st);
  }
  Choice c;
  if (!choose_kernel(h->dims, a.R, h->sm_count, a.route_only != 0, c)) return cudaErrorInvalidValue;
  h->last_kind = c.kind;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(h->sm_count);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = c.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, c.fn, a);
  if (prof) cudaEventRecord(e1, st);
  return e;
}

int common_checks(moe_handle* h, const uint16_t* x, int32_t rows, void* ws, size_t ws_bytes) {
  if (!h || !aligned16(x) || !ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOE_EINVAL;
  if (rows < 1 || rows > h->dims.max_rows) return MOE_EINVAL;
  if (ws_bytes < ws_layout(h->dims, rows).total) return MOE_EWORKSPACE;
  return MOE_OK;
}

void copy_layers(RoundArgs& a, const moe_layer_w* layers, int32_t L) {
  for (int32_t l = 0; l < L; ++l) {
    a.layer[l].router = layers[l].router;
    a.layer[l].gu_nib = layers[l].gateup_nib;
    a.layer[l].gu_sc = layers[l].gateup_scale;
    a.layer[l].dn_nib = layers[l].down_nib;
    a.layer[l].dn_sc = layers[l].down_scale;
    a.layer[l].slot = layers[l].slot_of_expert;
    a.layer[l].n_slots = layers[l].n_slots;
  }
}

}  // namespace

extern "C" {

int moe_create(const moe_dims* dims, int device, moe_handle** out) {
  if (!out) return MOE_EINVAL;
  *out = nullptr;
  int rc = check_dims(dims);
  if (rc != MOE_OK) return rc;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
    cudaGetLastError();
    return MOE_ECUDA;
  }
  DeviceGuard g(device);
  if (!g.ok) return MOE_ECUDA;
  int coop = 0, sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, device) != cudaSuccess || !coop) {
    cudaGetLastError();
    return MOE_ECUDA;
  }
  cudaError_t e = prepare_kernels(device, dims->hidden);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MOE_ECUDA;
  }
  if ((rc = check_plans(*dims, sms)) != MOE_OK) return rc;
  moe_handle* h = new moe_handle();
  h->dims = *dims;
  h->device = device;
  h->sm_count = sms;
  if (cudaMalloc(&h->status, sizeof(unsigned)) != cudaSuccess ||
      cudaMemset(h->status, 0, sizeof(unsigned)) != cudaSuccess) {
    cudaGetLastError();
    if (h->status) cudaFree(h->status);
    delete h;
    return MOE_ECUDA;
  }
  *out = h;
  return MOE_OK;
}

void moe_destroy(moe_handle* h) {
  if (!h) return;
  DeviceGuard g(h->device);
  if (h->gexec) cudaGraphExecDestroy(h->gexec);
  if (h->status) cudaFree(h->status);
  if (h->phase_ts) cudaFree(h->phase_ts);
  for (cudaEvent_t e : h->ev) cudaEventDestroy(e);
  delete h;
}

int moe_set_wait_limit_ns(moe_handle* h, uint64_t ns) {
  if (!h) return MOE_EINVAL;
  h->wait_ns = ns ? ns : kDefaultWaitNs;
  return MOE_OK;
}

int moe_set_tail_skip(moe_handle* h, int32_t rank) {
  if (!h || rank < 0) return MOE_EINVAL;
  h->tail_rank = rank;
  return MOE_OK;
}

int moe_route(moe_handle* h, const moe_layer_w* w, const uint16_t* x_bf16, int32_t rows,
              int32_t* topk_ids, float* topk_w, int32_t* union_ids, int32_t* n_union, void* ws,
              size_t ws_bytes, void* stream) {
  int rc = common_checks(h, x_bf16, rows, ws, ws_bytes);
  if (rc != MOE_OK) return rc;
  if (!w || !aligned16(w->router)) return MOE_EINVAL;
  DeviceGuard g(h->device);
  if (!g.ok) return MOE_ECUDA;
  RoundArgs a{};
  fill_args(a, h, rows, ws);
  a.L = 1;
  a.route_only = 1;
  a.x = x_bf16;
  a.user_ids = topk_ids;
  a.user_w = topk_w;
  a.user_union = union_ids;
  a.user_nunion = n_union;
  a.layer[0].router = w->router;
  h->last_launches = 1;
  return launch_round(h, a, static_cast<cudaStream_t>(stream), false) == cudaSuccess ? MOE_OK
                                                                                    : MOE_ECUDA;
}

int moe_decode_layer(moe_handle* h, const moe_layer_w* w, const uint16_t* x_bf16, int32_t rows,
                     float* out, void* ws, size_t ws_bytes, void* stream) {
  int rc = common_checks(h, x_bf16, rows, ws, ws_bytes);
  if (rc != MOE_OK) return rc;
  if ((rc = check_layer(w)) != MOE_OK) return rc;
  if (!aligned16(out)) return MOE_EINVAL;
  DeviceGuard g(h->device);
  if (!g.ok) return MOE_ECUDA;
  RoundArgs a{};
  fill_args(a, h, rows, ws);
  a.L = 1;
  a.x = x_bf16;
  a.out = out;
  copy_layers(a, w, 1);
  h->last_launches = 1;
  return launch_round(h, a, static_cast<cudaStream_t>(stream), false) == cudaSuccess ? MOE_OK
                                                                                    : MOE_ECUDA;
}

int moe_prefill_layer(moe_handle* h, const moe_layer_w* w, const uint16_t* x_bf16, int32_t tokens,
                      float* out, int32_t* expert_counts, void* ws, size_t ws_bytes, void* stream) {
  if (!h) return MOE_EINVAL;
  if (tokens < 1 || tokens > kMaxPrefillTokens || !aligned16(x_bf16) || !aligned16(out) || !aligned16(ws))
    return MOE_EINVAL;
  int rc = check_layer(w);
  if (rc != MOE_OK) return rc;
  if (expert_counts && (reinterpret_cast<uintptr_t>(expert_counts) & 3u)) return MOE_EINVAL;
  const PrefillWs L = prefill_ws_layout(h->dims, tokens);
  if (ws_bytes < L.total) return MOE_EWORKSPACE;
  DeviceGuard g(h->device);
  if (!g.ok) return MOE_ECUDA;
  char* base = static_cast<char*>(ws);
  PrefillArgs a{};
  a.H = h->dims.hidden;
  a.E = h->dims.n_experts;
  a.k = h->dims.top_k;
  a.I = h->dims.inter;
  a.T = tokens;
  a.x = x_bf16;
  a.out = out;
  a.router = w->router;
  a.gu_nib = w->gateup_nib;
  a.gu_sc = w->gateup_scale;
  a.dn_nib = w->down_nib;
  a.dn_sc = w->down_scale;
  a.slot = w->slot_of_expert;
  a.n_slots = w->n_slots;
  a.logits = reinterpret_cast<float*>(base + L.logits);
  a.ids = reinterpret_cast<int*>(base + L.ids);
  a.w = reinterpret_cast<float*>(base + L.w);
  a.counts = reinterpret_cast<int*>(base + L.counts);
  a.offs = reinterpret_cast<int*>(base + L.offs);
  a.cursor = reinterpret_cast<int*>(base + L.cursor);
  a.tiles_gu = reinterpret_cast<int*>(base + L.tiles_gu);
  a.tiles_dn = reinterpret_cast<int*>(base + L.tiles_dn);
  a.pos_tok = reinterpret_cast<int*>(base + L.pos_tok);
  a.pos_pick = reinterpret_cast<int*>(base + L.pos_pick);
  a.pick_pos = reinterpret_cast<int*>(base + L.pick_pos);
  a.hbuf = reinterpret_cast<uint16_t*>(base + L.hbuf);
  a.ybuf = reinterpret_cast<float*>(base + L.ybuf);
  a.user_counts = expert_counts;
  a.status = h->status;
  int launches = 0;
  const int e = prefill_launch(a, &launches, stream);
  h->last_launches = launches;
  return e == (int)cudaSuccess ? MOE_OK : MOE_ECUDA;
}

int moe_round(moe_handle* h, const moe_layer_w* layers, int32_t L, const uint16_t* x_bf16,
              int32_t rows, float* out, int32_t* stats, void* ws, size_t ws_bytes, int use_graph,
              void* stream) {
  int rc = common_checks(h, x_bf16, rows, ws, ws_bytes);
  if (rc != MOE_OK) return rc;
  if (!layers || L < 1 || !aligned16(out)) return MOE_EINVAL;
  if (L > kMaxLayers) return MOE_EUNSUPPORTED;
  for (int32_t l = 0; l < L; ++l)
    if ((rc = check_layer(&layers[l])) != MOE_OK) return rc;
  if (use_graph && !stream) return MOE_EINVAL;
  DeviceGuard g(h->device);
  if (!g.ok) return MOE_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  RoundArgs a{};
  fill_args(a, h, rows, ws);
  a.L = L;
  a.x = x_bf16;
  a.out = out;
  a.stats = stats;
  copy_layers(a, layers, L);
  if (!use_graph) {
    if (h->profiling && h->phase_ts) {
      a.phase_ts = h->phase_ts;
      h->phase_layers = L;
    }
    h->last_launches = 1;
    const cudaError_t e = launch_round(h, a, st, false);
    if (a.phase_ts) h->phase_kind = h->last_kind;
    return e == cudaSuccess ? MOE_OK : MOE_ECUDA;
  }
  GraphKey key;
  key.layers.assign(layers, layers + L);
  key.rows = rows;
  key.tail_rank = h->tail_rank;
  key.x = x_bf16;
  key.out = out;
  key.stats = stats;
  key.ws = ws;
  key.stream = stream;
  key.ws_bytes = ws_bytes;
  if (!h->gexec || !(key == h->gkey)) {
    if (h->gexec) {
      cudaGraphExecDestroy(h->gexec);
      h->gexec = nullptr;
    }
    if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
      return MOE_ECUDA;
    cudaError_t e = launch_round(h, a, st, true);
    cudaGraph_t graph = nullptr;
    cudaError_t e2 = cudaStreamEndCapture(st, &graph);
    if (e != cudaSuccess || e2 != cudaSuccess || !graph) {
      if (graph) cudaGraphDestroy(graph);
      cudaGetLastError();
      return MOE_ECUDA;
    }
    e = cudaGraphInstantiate(&h->gexec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) {
      h->gexec = nullptr;
      cudaGetLastError();
      return MOE_ECUDA;
    }
    h->gkey = key;
    h->graph_launches = 1;
  }
  if (cudaGraphLaunch(h->gexec, st) != cudaSuccess) return MOE_ECUDA;
  h->last_launches = h->graph_launches;
  return MOE_OK;
}

int moe_last_device_status(moe_handle* h, void* stream) {
  if (!h) return MOE_EINVAL;
  DeviceGuard g(h->device);
  if (!g.ok) return MOE_ECUDA;
  unsigned v = 0;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ECUDA;
  if (cudaMemcpy(&v, h->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ECUDA;
  if (cudaMemset(h->status, 0, sizeof(unsigned)) != cudaSuccess) return MOE_ECUDA;
  if (v & kStatusTimeout) return MOE_ETIMEOUT;
  return (v & kStatusBadSlot) ? MOE_EINVAL : MOE_OK;
}

int32_t moe_last_launch_count(const moe_handle* h) { return h ? h->last_launches : 0; }

int moe_profile(moe_handle* h, int enable) {
  if (!h) return MOE_EINVAL;
  h->profiling = enable != 0;
  h->ev_used = 0;
  h->phase_layers = 0;
  if (h->profiling && !h->phase_ts) {
    DeviceGuard g(h->device);
    if (!g.ok) return MOE_ECUDA;
    const size_t n = (size_t)kMaxLayers * kPhases * h->sm_count;
    if (cudaMalloc(&h->phase_ts, n * sizeof(long long)) != cudaSuccess) {
      cudaGetLastError();
      h->phase_ts = nullptr;
      return MOE_ECUDA;
    }
  }
  return MOE_OK;
}

int moe_profile_read(moe_handle* h, int kind, double* total_ms, int32_t* launches) {
  if (!h || !total_ms || !launches || kind != 0) return MOE_EINVAL;
  DeviceGuard g(h->device);
  if (!g.ok) return MOE_ECUDA;
  double t = 0.0;
  int32_t n = 0;
  for (size_t i = 0; i + 1 < h->ev_used; i += 2) {
    if (cudaEventSynchronize(h->ev[i + 1]) != cudaSuccess) return MOE_ECUDA;
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, h->ev[i], h->ev[i + 1]) != cudaSuccess) return MOE_ECUDA;
    t += ms;
    ++n;
  }
  *total_ms = t;
  *launches = n;
  return MOE_OK;
}

int moe_profile_phases(moe_handle* h, double* mean_us, double* max_us, int32_t n_phases) {
  if (!h || !mean_us || !max_us) return MOE_EINVAL;
  if (!h->phase_ts || h->phase_layers < 1) return MOE_EINVAL;
  const int stamps = h->phase_kind == kKindWide ? kPhases : kSplitPhases;
  if (n_phases < stamps - 1) return MOE_EINVAL;
  DeviceGuard g(h->device);
  if (!g.ok) return MOE_ECUDA;
  const int G = h->sm_count, L = h->phase_layers;
  // the stamps are SM cycle counts (differences within one CTA); cycles -> us at the
  // SM clock the device reports
  int khz = 0;
  if (cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, h->device) != cudaSuccess || khz <= 0) return MOE_ECUDA;
  const double us_per_cycle = 1e3 / (double)khz;
  std::vector<long long> ts((size_t)L * stamps * G);
  if (cudaDeviceSynchronize() != cudaSuccess ||
      cudaMemcpy(ts.data(), h->phase_ts, ts.size() * sizeof(long long), cudaMemcpyDeviceToHost) !=
          cudaSuccess)
    return MOE_ECUDA;
  for (int p = 0; p + 1 < stamps; ++p) {
    double sum = 0.0, mx = 0.0;
    for (int l = 0; l < L; ++l) {
      double lmax = 0.0;
      for (int c = 0; c < G; ++c) {
        const double d = (double)(ts[((size_t)l * stamps + p + 1) * G + c] -
                                  ts[((size_t)l * stamps + p) * G + c]) * us_per_cycle;
        sum += d;
        if (d > lmax) lmax = d;
      }
      mx += lmax;
    }
    mean_us[p] = sum / ((double)L * G);
    max_us[p] = mx / L;
  }
  return stamps - 1;
}

}  // extern "C"

// =====================================================================================
// Allocation-free variant of moe_decode_layer.
//
// Some callers cannot allocate device memory at all: code that runs inside another
// framework's memory pool with allocation disabled, allocation-free real-time or
// embedded loops, or hosts that forbid cudaMalloc after start-up.  For them the
// workspace (grid-barrier words, router logits, exchanged SwiGLU outputs, output
// accumulators) lives in the file-scope array below, which the CUDA runtime places on
// every device that loads this library and keeps until the process exits.  The caller
// passes only inputs, outputs and a status word; this path calls no cudaMalloc, cudaFree
// or allocating library routine.

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)8 << 20;  // 8 MiB per device
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDevice {
  bool ready = false;
  void* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int sms = 0;
};

NoAllocDevice g_noalloc[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;

// One-time set-up of the current device: the device address of the scratch array (in
// host code the symbol names a host-side stand-in, not device memory), the SM count,
// and the kernels' shared-memory limits.
int noalloc_setup(int dev, NoAllocDevice** out) {
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocDevice& d = g_noalloc[dev];
  if (!d.ready) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return MOE_ECUDA;
    }
    int sms = 0, coop = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop) {
      cudaGetLastError();
      return MOE_ECUDA;
    }
    if (prepare_kernels(dev, 256) != cudaSuccess || prepare_kernels(dev, kMaxHidden) != cudaSuccess) {
      cudaGetLastError();
      return MOE_ECUDA;
    }
    d.scratch = p;
    d.sms = sms;
    d.ready = true;
  }
  *out = &d;
  return MOE_OK;
}

}  // namespace

extern "C" int moe_decode_layer_noalloc(const moe_dims* dims, const moe_layer_w* w,
                                        const uint16_t* x_bf16, int32_t rows, float* out,
                                        unsigned* dev_status, void* stream) {
  int rc = check_dims(dims);
  if (rc != MOE_OK) return rc;
  if ((rc = check_layer(w)) != MOE_OK) return rc;
  if (!aligned16(x_bf16) || !aligned16(out) || rows < 1 || rows > dims->max_rows) return MOE_EINVAL;
  // the status word is where a kernel reports what it found; without it errors are lost
  if (!dev_status || (reinterpret_cast<uintptr_t>(dev_status) & 3u)) return MOE_EINVAL;
  const WsLayout L = ws_layout(*dims, rows);
  if (L.total > kNoAllocScratchBytes) return MOE_EWORKSPACE;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) {
    cudaGetLastError();
    return MOE_ECUDA;
  }
  NoAllocDevice* d = nullptr;
  if ((rc = noalloc_setup(dev, &d)) != MOE_OK) return rc;
  Choice c;
  if (!choose_kernel(*dims, rows, d->sms, false, c) ||
      (size_t)((dims->n_experts + d->sms - 1) / d->sms) * dims->hidden * 4 > (size_t)64 * 1024)
    return MOE_EUNSUPPORTED;
  char* ws = static_cast<char*>(d->scratch);
  RoundArgs a{};
  const moe_dims& dd = *dims;
  a.H = dd.hidden;
  a.E = dd.n_experts;
  a.k = dd.top_k;
  a.I = dd.inter;
  a.R = rows;
  a.Rmax = dd.max_rows;
  a.L = 1;
  a.bar = reinterpret_cast<unsigned*>(ws + L.ctrl);
  a.logits = reinterpret_cast<float*>(ws + L.logits);
  a.hbuf = reinterpret_cast<float*>(ws + L.hbuf);
  a.acc = reinterpret_cast<unsigned long long*>(ws + L.acc);
  a.status = dev_status;
  a.wait_cycles = kDefaultWaitCycles;
  a.x = x_bf16;
  a.out = out;
  copy_layers(a, w, 1);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the barrier words must start at zero; logits, h and the accumulators are written
  // (the accumulators cleared) by the kernel itself
  if (cudaMemsetAsync(a.bar, 0, 256, st) != cudaSuccess) return MOE_ECUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(d->sms);
  cfg.blockDim = dim3(NT);
  cfg.dynamicSmemBytes = c.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, c.fn, a);
  return e == cudaSuccess ? MOE_OK : MOE_ECUDA;
}
