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
// (exchanged between CTAs by the tensor-core kernel: one row per routed (row, expert)
// pair, grouped by expert, as bf16 hi + lo in fragment order), and the split kernel's
// output accumulators [2 (layer parity)][kAccCopies][rows][H] (int64, 2^32-scaled).
constexpr int kAccCopies = 8;
struct WsLayout {
  size_t ctrl, logits, hbuf, acc, total;
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

// Prefill-width layer (moe_prefill.cu): tokens per call, device arguments, workspace.
constexpr int kMaxPrefillTokens = 65536;

struct PrefillArgs {
  int H, E, k, I, T;
  const uint16_t* x;  // [T][H] bf16 bits
  float* out;         // [T][H]
  const float* router;
  const uint8_t* gu_nib;
  const uint16_t* gu_sc;
  const uint8_t* dn_nib;
  const uint16_t* dn_sc;
  const int32_t* slot;  // expert -> bank slot, or null
  int n_slots;
  // workspace
  float* logits;     // [T][E]
  int* ids;          // [T*k] expert of pick t*k + j (rank order)
  float* w;          // [T*k] renormalised weight of each pick
  int* counts;       // [E] picks per expert
  int* offs;         // [E+1] start of each expert's run of positions
  int* cursor;       // [E] scatter cursors
  int* tiles_gu;     // [E+1] prefix of gate/up token tiles per expert
  int* tiles_dn;     // [E+1] prefix of down token tiles per expert
  int* pos_tok;      // [T*k] token at each position
  int* pos_pick;     // [T*k] pick at each position
  int* pick_pos;     // [T*k] position of each pick
  uint16_t* hbuf;    // [T*k][I] h' as bf16 hi + lo in the down operand order
  float* ybuf;       // [T*k][H] down output of each position
  int* user_counts;  // [E] or null
  unsigned* status;
};

// Byte offsets of the prefill workspace regions (each 256-aligned).
struct PrefillWs {
  size_t logits, ids, w, counts, offs, cursor, tiles_gu, tiles_dn, pos_tok, pos_pick, pick_pos, hbuf,
      ybuf, total;
};
PrefillWs prefill_ws_layout(const moe_dims& d, int tokens);

// Enqueues the prefill kernels on `stream` (a cudaStream_t); returns a cudaError_t code
// and the number of kernels launched.
int prefill_launch(const PrefillArgs& a, int* launches, void* stream);

// Per-expert packed sizes (bytes).
inline size_t gu_nib_bytes(const moe_dims& d) { return (size_t)d.inter * d.hidden; }
inline size_t gu_sc_bytes(const moe_dims& d) { return (size_t)d.inter * d.hidden / 8; }
inline size_t dn_nib_bytes(const moe_dims& d) { return (size_t)d.inter * d.hidden / 2; }
inline size_t dn_sc_bytes(const moe_dims& d) { return (size_t)d.inter * d.hidden / 16; }

}  // namespace moe
