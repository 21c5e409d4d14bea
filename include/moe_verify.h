/*
 * moe_verify.h -- C ABI of the MoE layer of a speculative-decoding verify round,
 * on one NVIDIA GB300 (sm_103a).
 *
 * The layer (sources: "How AlphaInfer makes local decoding fast", sections 2 and 3.1:
 * a decode round over 1..16 token rows replayed as one captured graph with
 * per-request data as ingress buffers, where every extra verified row can route to
 * experts the other rows did not need and so adds weight bytes; "infero", the
 * decoder-block diagram and Design notes: a SwiGLU expert FFN silu(W_g x) * (W_u x)
 * -> W_d, weights consumed in 32-element block encoding, block scales folded in in
 * float; a dedicated top-k routing kernel at decode):
 *
 *   1. logits[r][e] = Wr[e] . x[r]                  fp32, fixed summation order (*)
 *   2. per row: the k largest logits, ordered by (logit desc, id asc);
 *      w_j = exp(l_j - l_1) / sum_i exp(l_i - l_1)   (softmax renormalised over the k)
 *   3. U = ascending distinct ids over all rows (each routed expert's weights are
 *      streamed once per call, however many rows picked it)
 *   4. per (row, routed expert): h = silu(Wg x) * (Wu x), silu(t) = t / (1 + e^-t)
 *   5. out[r] = sum_j w_j * (Wd h_{r,j})            (j in rank order)
 * Expert weights are int4 codes q in [-8, 7] with one fp16 scale per 32 codes;
 * weight = scale * q.  Activations in are bf16; everything after is fp32.
 *
 * (*) The router summation order is part of the definition so that the top-k
 * decision is reproducible bit for bit: 32 lane partials, lane l takes elements
 * 128c + 4l + j (c ascending, j = 0..3), each with one correctly rounded fma; the
 * partials are combined by p_l <- p_l + p_{l^o} for o = 16, 8, 4, 2, 1; logit = p_0.
 *
 * Conventions for every call below:
 *   - Device pointers are caller-owned device memory, 16-byte aligned (256 recommended).
 *     The library never frees caller memory.  Host pointers are plain host memory.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Compute calls are
 *     asynchronous on that stream and return only argument/launch status; errors a
 *     kernel finds (a bounded wait that gave up) are read with moe_last_device_status.
 *   - Return codes: MOE_OK, or a negative MOE_E* code; moe_strerror names it.
 *   - Rows are independent: a row's outputs do not depend on which other rows share
 *     the call or on its position among them (bitwise).
 *   - Activations must be finite with |x| < 2^40 (and so must the SwiGLU output h);
 *     beyond that range results are undefined.
 *   - Rounds of fewer than 13 rows evaluate each 32-element block dot of steps 4 and 5
 *     exactly in integers, from the block's codes and its activations in block fixed
 *     point (x: 16 bits relative to the block's largest |x|; h: 23 bits), then scale it
 *     in fp32; the rounding of the smaller activations of a block (at most 2^-15 and
 *     2^-22 of the block's largest) stays within the stated output tolerance.  Wider
 *     rounds use bf16 x (exact) and h split into bf16 hi + lo on the tensor cores.
 *   - Every contribution to a row's output (rounds of fewer than 13 rows: one expert
 *     and 32-element slice of the intermediate dimension; wider rounds: one expert and
 *     chunk of up to 768 intermediate elements) is added as round(y * 2^32) into 64-bit
 *     integer accumulators, so the sum is exact and independent of the order of the
 *     adds; every such contribution and every output must stay below 2^31 in magnitude
 *     (beyond that results are undefined).
 */
#ifndef MOE_VERIFY_H
#define MOE_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  MOE_OK = 0,
  MOE_EINVAL = -1,       /* bad dimensions, NULL or misaligned pointer, rows out of range */
  MOE_ECUDA = -2,        /* a CUDA runtime call failed (no device, launch failure, ...) */
  MOE_EWORKSPACE = -3,   /* workspace smaller than moe_workspace_bytes() */
  MOE_ETIMEOUT = -4,     /* a device-side bounded wait gave up (moe_last_device_status) */
  MOE_EUNSUPPORTED = -5  /* valid dimensions this build does not handle (see moe_create) */
};

/* which matrix set a packing call refers to */
enum { MOE_GATEUP = 0, MOE_DOWN = 1 };

/* Layer dimensions.  hidden H, n_experts E, top_k k, inter I (expert intermediate),
 * max_rows = the largest row count any call on this handle will pass. */
typedef struct moe_dims {
  int32_t hidden, n_experts, top_k, inter, max_rows;
} moe_dims;

/* One layer's weights, all DEVICE pointers in the packed layout of moe_pack_q4:
 *   router        fp32 [E][H] row-major
 *   gateup_nib    E * moe_packed_bytes(MOE_GATEUP, 0) bytes
 *   gateup_scale  E * moe_packed_bytes(MOE_GATEUP, 1) bytes of fp16 bits
 *   down_nib      E * moe_packed_bytes(MOE_DOWN, 0) bytes
 *   down_scale    E * moe_packed_bytes(MOE_DOWN, 1) bytes of fp16 bits          */
typedef struct moe_layer_w {
  const float* router;
  const uint8_t* gateup_nib;
  const uint16_t* gateup_scale;
  const uint8_t* down_nib;
  const uint16_t* down_scale;
  /* Expert -> slot indirection (AlphaInfer docs, section 2: "which expert lives where"
   * is per-round ingress data written into fixed buffers; section 5.1: one shared slot
   * bank across layers).  NULL: expert e's packed weights are entry e of the four
   * arrays above (as moe_pack_q4 writes them for a layer).  Otherwise a DEVICE int32
   * array [n_experts]: expert e's weights are entry slot_of_expert[e] of a bank of
   * n_slots entries that the four pointers address (one moe_pack_q4 entry per slot;
   * several layers may share one bank).  The kernel reads the table during the call,
   * so a captured round (moe_round with use_graph) picks up new table contents
   * without being rebuilt.  A slot outside [0, n_slots) is not read: the layer
   * computes with slot 0 instead and moe_last_device_status returns MOE_EINVAL. */
  const int32_t* slot_of_expert;
  int32_t n_slots;
} moe_layer_w;

typedef struct moe_handle moe_handle;

/* Validates dims and binds a handle to `device` (queries its SM count, allocates a
 * 4-byte device status word -- the only device allocation the library makes).
 * Supported: hidden a multiple of 256 in [256, 2048], inter a multiple of 256 in
 * [256, 4096], 1 <= top_k <= min(n_experts, 32), n_experts <= 512, 1 <= max_rows <= 32
 * (and the shared-memory plan must fit one SM).
 * MOE_EINVAL for dims that make no sense, MOE_EUNSUPPORTED for sizes outside those
 * ranges, MOE_ECUDA if the device cannot be used.  *out is NULL on failure. */
int moe_create(const moe_dims* dims, int device, moe_handle** out);
void moe_destroy(moe_handle* h);

/* Device workspace (bytes) a call with `rows` rows needs: barrier words, router logits,
 * the SwiGLU outputs exchanged between CTAs by the tensor-core path and the output
 * accumulators (2 x 8 copies x rows x H int64; the tensor-core path uses one copy).  It depends only on
 * the dimensions and the row count, so it takes the dimensions rather than a handle and
 * can be sized before any handle exists.  0 for invalid dims/rows. */
size_t moe_workspace_bytes(const moe_dims* dims, int32_t rows);

/* Packed size of ONE expert: part 0 = code bytes, part 1 = scale bytes (codes and scales
 * are separate device arrays, so each has its own size).  0 if invalid. */
size_t moe_packed_bytes(const moe_dims* dims, int which, int part);

/* Host-side packer (HOST buffers).  Packs n_experts consecutive experts:
 *   MOE_GATEUP: q_a = gate codes [n][I][H], s_a = gate scales [n][I][H/32],
 *               q_b = up codes [n][I][H],   s_b = up scales [n][I][H/32]
 *   MOE_DOWN:   q_a = down codes [n][H][I], s_a = down scales [n][H][I/32]; q_b, s_b unused
 * into nib_out / scale_out (n * moe_packed_bytes(which, 0 / 1) bytes).  Codes outside
 * [-8, 7] give MOE_EINVAL.  Layout (32-element blocks, code q stored as the nibble
 * q + 8, element 2t in the low nibble of byte t of its block):
 *   gate/up codes  [E][I][2: gate, up][H/32 blocks][16 B]   (intermediate row i of an
 *   gate/up scales [E][I][2][H/32]                           expert: gate, then up)
 *   down codes     [E][I/32 blocks][H rows][16 B]            (block-major: block b of all
 *   down scales    [E][I/32][H]                               H output rows is one run)
 * where, within each gate/up row, the code block and the scale of logical block b are
 * stored at position b ^ (i & 7) (i the row's intermediate index; gate and up alike).
 * Down block b of output row o is at b * H + o. */
int moe_pack_q4(const moe_dims* dims, int which, int32_t n_experts, const int8_t* q_a,
                const uint16_t* s_a, const int8_t* q_b, const uint16_t* s_b, uint8_t* nib_out,
                uint16_t* scale_out);

/* Steps 1-3 only (router GEMV, top-k + renormalised weights, union).
 * x_bf16 [rows][H] device; topk_ids [rows][k] int32 (rank order), topk_w [rows][k]
 * fp32, union_ids [E] int32 (first *n_union valid, ascending), n_union: device int32.
 * Any of the four outputs may be NULL.  ws: device workspace of ws_bytes. */
int moe_route(moe_handle* h, const moe_layer_w* w, const uint16_t* x_bf16, int32_t rows,
              int32_t* topk_ids, float* topk_w, int32_t* union_ids, int32_t* n_union, void* ws,
              size_t ws_bytes, void* stream);

/* Steps 1-5 for one layer.  x_bf16 [rows][H] device, out [rows][H] fp32 device. */
int moe_decode_layer(moe_handle* h, const moe_layer_w* w, const uint16_t* x_bf16, int32_t rows,
                     float* out, void* ws, size_t ws_bytes, void* stream);

/* A round over an L-layer stack, layer after layer in stream order (layer l+1's
 * routing starts only after layer l's output is complete).  layers: HOST array [L] of
 * device weight sets; x_bf16 [L][rows][H] device (layer l reads its own rows);
 * out [L][rows][H] fp32 device; stats: device int32 [L] receiving |U| per layer, or
 * NULL.  use_graph != 0 captures the round once per (handle, argument set) into a
 * CUDA graph and replays it on later calls with the same arguments; the buffers
 * are ingress: write new rows into the same x buffer and call again.  use_graph
 * needs a non-default stream. */
int moe_round(moe_handle* h, const moe_layer_w* layers, int32_t L, const uint16_t* x_bf16,
              int32_t rows, float* out, int32_t* stats, void* ws, size_t ws_bytes, int use_graph,
              void* stream);

/* moe_round with the rows in and the outputs out in HOST memory: on `stream`, in this
 * order, the copy of x_host into x_dev, the round (moe_round on x_dev / out_dev), and the
 * copy of out_dev into out_host -- what a caller holding the draft rows on the host runs
 * once per verify round (AlphaInfer docs §2: the round's rows are ingress into one
 * captured round).
 *   - dims: the dims the handle was created with (the copies move L * rows * hidden
 *     elements); call with the handle's device current.
 *   - x_host [L][rows][H] bf16 bits and out_host [L][rows][H] fp32, host memory owned
 *     by the caller.  Page-locked memory makes both copies asynchronous; with pageable
 *     memory the calling thread waits for each copy.
 *   - x_dev [L][rows][H] and out_dev [L][rows][H]: the caller's device staging buffers
 *     (16-byte aligned); they are moe_round's x_bf16 and out, so with use_graph the
 *     round replays while they, ws and stream stay the same.
 *   - stats, ws, ws_bytes, use_graph, stream: as for moe_round.
 *   - sync != 0: returns after the stream has finished, with out_host written, and with
 *     moe_last_device_status's answer (MOE_ETIMEOUT or MOE_EINVAL if the kernel raised
 *     one, the status word cleared).  sync == 0: returns once the work is enqueued; the
 *     caller synchronizes the stream before reading out_host and may read the status
 *     with moe_last_device_status.
 * Allocates nothing.  Nothing is enqueued when an argument is wrong: MOE_EINVAL for a
 * NULL handle, dims, layers or buffer, L outside [1, 128] or rows outside [1, max_rows],
 * moe_create's code for dims it would reject.  Otherwise moe_round's codes for the
 * round (the rows' copy is then already enqueued) and MOE_ECUDA if a copy fails. */
int moe_round_host(moe_handle* h, const moe_dims* dims, const moe_layer_w* layers, int32_t L,
                   const uint16_t* x_host, int32_t rows, float* out_host, uint16_t* x_dev,
                   float* out_dev, int32_t* stats, void* ws, size_t ws_bytes, int use_graph, int sync,
                   void* stream);

/* Prefill-width layer: steps 1-5 for many token rows at once (a prompt's tokens), the
 * infero README's MoE prefill path ("Beyond plain text decode": a counting sort of the
 * (token, expert) picks by expert, then one GEMM per expert).  Same weights, routing
 * (canonical router order, ties to the lower id, renormalised top-k weights) and
 * output definition as moe_decode_layer, for 1 <= tokens <= 65536:
 *   out[t] = sum_j w_{t,j} Wd_{e_j} (silu(Wg_{e_j} x_t) * (Wu_{e_j} x_t)).
 * Gate/up and down run on the tensor cores (bf16 operands that are exact for the int4
 * codes and the bf16 rows, fp32 accumulation per 32-element block, h' split into bf16
 * hi + lo), so a token's output equals moe_decode_layer's within the layer tolerance,
 * not bitwise; it does not depend on the other tokens of the call.
 * x_bf16 [tokens][H] device, out [tokens][H] fp32 device (both 16-byte aligned);
 * expert_counts: device int32 [E] receiving the picks per expert, or NULL.
 * ws: device workspace (16-byte aligned) of at least moe_prefill_workspace_bytes.
 * The handle's max_rows does not limit tokens.  MOE_EINVAL for bad arguments,
 * MOE_EWORKSPACE for a short workspace; slot-table entries outside the bank are
 * reported by moe_last_device_status.  Enqueues 7 kernels and one memset. */
size_t moe_prefill_workspace_bytes(const moe_dims* dims, int32_t tokens);
int moe_prefill_layer(moe_handle* h, const moe_layer_w* w, const uint16_t* x_bf16, int32_t tokens,
                      float* out, int32_t* expert_counts, void* ws, size_t ws_bytes, void* stream);

/* Synchronizes `stream`, reads and clears the handle's device status word.
 * MOE_OK, MOE_ETIMEOUT (a bounded device wait gave up), MOE_EINVAL (a slot table entry
 * was outside [0, n_slots)), or MOE_ECUDA. */
int moe_last_device_status(moe_handle* h, void* stream);

/* Number of kernel launches the most recent moe_route / moe_decode_layer /
 * moe_round / moe_prefill_layer call enqueued (a graph replay counts the kernels
 * inside it). */
int32_t moe_last_launch_count(const moe_handle* h);

/* Bound on every device-side wait of this handle's kernels (default 2 s; 0 restores
 * the default).  A tiny bound makes the waits give up at once: the kernels then set
 * the timeout bit, drain their copies in flight under the default bound, and return,
 * so tests can exercise the MOE_ETIMEOUT path without any hang. */
int moe_set_wait_limit_ns(moe_handle* h, uint64_t ns);

/* Routing tail skip (an approximation; off by default).  Avalon README, "Numbers" (RX
 * 7900 XT): experts that every token of a verification routes only at rank 7 or lower
 * are skipped.  With rank = T > 0, every later moe_route / moe_decode_layer / moe_round
 * call of this handle drops a union expert when each row that picked it has it at
 * 1-based rank >= T (T = 7 is the page's setting): the expert leaves the union
 * (union_ids, n_union and stats shrink), its picks contribute nothing to the output,
 * and the remaining weights are not renormalised (the page does not say; this is the
 * reading taken).  topk_ids / topk_w still report every row's k picks.  rank = 0 turns
 * it off; T = 1 drops every expert (output 0); T > k drops none.  Returns MOE_EINVAL for
 * a NULL handle or rank < 0.  moe_decode_layer_noalloc never skips. */
int moe_set_tail_skip(moe_handle* h, int32_t rank);

/* Timing of eager (non-graph) calls.  moe_profile(h, 1) starts recording a CUDA event
 * pair around every kernel launch the handle makes on the caller's stream, and
 * per-phase device timestamps inside moe_round (first use allocates a small device
 * buffer for them); earlier records are discarded.  moe_profile(h, 0) stops.
 * moe_profile_read synchronizes the events and returns the summed device time in ms
 * and the launch count (kind must be 0: the fused round kernel).
 * moe_profile_phases writes, for the last profiled moe_round, the mean over CTAs and
 * layers (mean_us) and the per-layer maximum over CTAs averaged over layers (max_us)
 * of its phases and returns how many it wrote (or a negative MOE_E* code); n_phases
 * >= 12 always suffices.  Rounds of fewer than 13 rows (10 phases): router GEMV,
 * logits barrier (and the previous layer's output written), routing, piece issue, wait
 * for the first gate/up bytes, units before the last, the last unit's gate/up, its
 * SwiGLU and the wait for its down bytes, its down products, layer-end barrier.  Wider rounds (12 phases): router GEMV,
 * barrier 1 (and the previous layer's output written), routing, wait for the first
 * staged gate/up chunk, gate/up until the last chunk has landed, gate/up after it,
 * barrier 2, (zero), down pass, (zero), (zero), barrier 3. */
int moe_profile(moe_handle* h, int enable);
int moe_profile_read(moe_handle* h, int kind, double* total_ms, int32_t* launches);
int moe_profile_phases(moe_handle* h, double* mean_us, double* max_us, int32_t n_phases);

/* Allocation-free moe_decode_layer, for callers that may not allocate device memory at
 * all (allocation disabled by a surrounding memory pool, allocation-free real-time
 * loops, hosts that forbid cudaMalloc after start-up).  There is no counterpart on the
 * pages this layer follows; it is an integration convenience.
 *   - Needs no handle and no workspace: the scratch (barrier words, logits, exchanged
 *     SwiGLU outputs, output accumulators) is one static device array of
 *     MOE_NOALLOC_SCRATCH_BYTES that every device loading this library holds until the
 *     process exits.
 *   - Runs on the current device.  Its first call on a device sets that device up
 *     (looks up the array's device address, the SM count, the kernels' shared-memory
 *     limits); make that first call before any stream capture on the device.
 *   - Arguments as for moe_decode_layer, plus dev_status: a caller-owned device word
 *     (required; NULL gives MOE_EINVAL) into which the kernel ORs what it finds: bit 1
 *     (value 1) if a bounded device wait gave up (the output is then incomplete), bit 2
 *     (value 2) if an expert-table entry was outside [0, n_slots) (slot 0 was used
 *     instead).  The caller clears the word and reads it after the stream has finished.
 *     Returns MOE_EWORKSPACE if the layer needs more scratch than the array holds
 *     (moe_workspace_bytes(dims, rows) > MOE_NOALLOC_SCRATCH_BYTES).
 *   - Calls no cudaMalloc, cudaFree or allocating routine.  Every call shares the one
 *     array: calls whose executions overlap on the GPU (different streams, or different
 *     host threads without ordering) race on it and give wrong results. */
#define MOE_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)
int moe_decode_layer_noalloc(const moe_dims* dims, const moe_layer_w* w, const uint16_t* x_bf16,
                             int32_t rows, float* out, unsigned* dev_status, void* stream);

const char* moe_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* MOE_VERIFY_H */
