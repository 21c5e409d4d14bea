// Internal declarations shared by the host code and the CUDA launchers of the
// verify-round MoE library.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/moe_verify.h"

namespace moe {

constexpr int kMaxRows = 32;   // rows are tracked in 32-bit masks
constexpr int kMaxExperts = 512;   // routing keeps 16 logits per lane in registers
constexpr int kMaxTopK = 32;
constexpr int kMinHidden = 256, kMaxHidden = 2048;
constexpr int kMaxInter = 4096;
constexpr int kMaxLayers = 128;  // layers per moe_round call (weight table travels as kernel parameters)

// 0 = valid and supported, MOE_EINVAL, or MOE_EUNSUPPORTED.
int check_dims(const moe_dims* d);

// Byte offsets of the workspace regions for `rows` rows (each region 256-aligned):
// grid-barrier words, router logits [rows][E], weighted SwiGLU outputs h' [rows*k][I]
// (fp32, one row per routed (row, expert) pair, grouped by expert, in the kernel's
// operand-pair order).
struct WsLayout {
  size_t ctrl, logits, hbuf, total;
};
WsLayout ws_layout(const moe_dims& d, int rows);

#ifdef __CUDACC__
#define MOE_HD __host__ __device__
#else
#define MOE_HD
#endif

// Packed rows store their 32-element blocks permuted: logical block b sits at position
// b ^ (key & 7), codes and scales alike (rows have a multiple of 8 blocks); the key is
// the output row o of a down row and the intermediate index i of a gate/up row (gate
// and up of one i share it).  The same logical block of 8 consecutive down rows, or of
// the gate/up rows of 4 consecutive units, then falls in 8 (4) different 16-byte bank
// groups of shared memory, so the tensor-core fragment loads of one block of 8 rows
// have no (at most 2-way) bank conflicts; a warp reading the blocks of one row (lane
// per block) reads a permutation of them, conflict-free.
MOE_HD inline int block_pos(int b, int key) { return b ^ (key & 7); }

// Per-expert packed sizes (bytes).
inline size_t gu_nib_bytes(const moe_dims& d) { return (size_t)d.inter * d.hidden; }
inline size_t gu_sc_bytes(const moe_dims& d) { return (size_t)d.inter * d.hidden / 8; }
inline size_t dn_nib_bytes(const moe_dims& d) { return (size_t)d.inter * d.hidden / 2; }
inline size_t dn_sc_bytes(const moe_dims& d) { return (size_t)d.inter * d.hidden / 16; }

}  // namespace moe
