// Host-side parts of the verify-round MoE library: dimension checks, workspace and
// packed sizes, the int4 block packer, error strings (none of these touch a GPU), and
// the host-buffer round (stream-ordered copies around moe_round).
#include <cstring>

#include <cuda_runtime.h>

#include "moe_internal.h"

namespace moe {

int check_dims(const moe_dims* d) {
  if (!d) return MOE_EINVAL;
  if (d->hidden <= 0 || d->n_experts <= 0 || d->top_k <= 0 || d->inter <= 0 || d->max_rows <= 0)
    return MOE_EINVAL;
  if (d->top_k > d->n_experts) return MOE_EINVAL;
  if (d->hidden % 128 || d->inter % 32) return MOE_EINVAL;  // block and router-order structure
  if (d->hidden % 256 || d->hidden < kMinHidden || d->hidden > kMaxHidden) return MOE_EUNSUPPORTED;
  if (d->inter % 256) return MOE_EUNSUPPORTED;  // 16-byte aligned bulk copies of scale rows
  if (d->inter > kMaxInter || d->n_experts > kMaxExperts || d->top_k > kMaxTopK ||
      d->max_rows > kMaxRows)
    return MOE_EUNSUPPORTED;
  return MOE_OK;
}

static size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

WsLayout ws_layout(const moe_dims& d, int rows) {
  WsLayout L{};
  size_t R = (size_t)rows, E = (size_t)d.n_experts, k = (size_t)d.top_k;
  size_t off = 0;
  L.ctrl = off;     off += 256;
  L.logits = off;   off += up256(R * E * 4);
  L.hbuf = off;     off += up256(R * k * (size_t)d.inter * 4);
  L.acc = off;      off += up256((size_t)2 * kAccCopies * R * (size_t)d.hidden * 8);
  L.total = off;
  return L;
}

PrefillWs prefill_ws_layout(const moe_dims& d, int tokens) {
  const size_t T = (size_t)tokens, E = (size_t)d.n_experts, P = T * (size_t)d.top_k;
  PrefillWs w{};
  size_t off = 0;
  w.logits = off;   off += up256(T * E * 4);
  w.ids = off;      off += up256(P * 4);
  w.w = off;        off += up256(P * 4);
  w.counts = off;   off += up256(E * 4);
  w.offs = off;     off += up256((E + 1) * 4);
  w.cursor = off;   off += up256(E * 4);
  w.tiles_gu = off; off += up256((E + 1) * 4);
  w.tiles_dn = off; off += up256((E + 1) * 4);
  w.pos_tok = off;  off += up256(P * 4);
  w.pos_pick = off; off += up256(P * 4);
  w.pick_pos = off; off += up256(P * 4);
  w.hbuf = off;     off += up256(P * (size_t)d.inter * 4);
  w.ybuf = off;     off += up256(P * (size_t)d.hidden * 4);
  w.total = off;
  return w;
}

}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_workspace_bytes(const moe_dims* dims, int32_t rows) {
  if (check_dims(dims) != MOE_OK || rows < 1 || rows > dims->max_rows) return 0;
  return ws_layout(*dims, rows).total;
}

size_t moe_prefill_workspace_bytes(const moe_dims* dims, int32_t tokens) {
  if (check_dims(dims) != MOE_OK || tokens < 1 || tokens > kMaxPrefillTokens) return 0;
  return prefill_ws_layout(*dims, tokens).total;
}

size_t moe_packed_bytes(const moe_dims* dims, int which, int part) {
  if (check_dims(dims) != MOE_OK || (part != 0 && part != 1)) return 0;
  if (which == MOE_GATEUP) return part == 0 ? gu_nib_bytes(*dims) : gu_sc_bytes(*dims);
  if (which == MOE_DOWN) return part == 0 ? dn_nib_bytes(*dims) : dn_sc_bytes(*dims);
  return 0;
}

// One 32-element block of codes -> 16 bytes: element 2t in the low nibble of byte t,
// element 2t+1 in the high nibble, each stored as q + 8.
static bool pack_block(const int8_t* q, uint8_t* dst) {
  for (int t = 0; t < 16; ++t) {
    int lo = q[2 * t], hi = q[2 * t + 1];
    if (lo < -8 || lo > 7 || hi < -8 || hi > 7) return false;
    dst[t] = (uint8_t)((lo + 8) | ((hi + 8) << 4));
  }
  return true;
}

int moe_pack_q4(const moe_dims* dims, int which, int32_t n_experts, const int8_t* q_a,
                const uint16_t* s_a, const int8_t* q_b, const uint16_t* s_b, uint8_t* nib_out,
                uint16_t* scale_out) {
  int rc = check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (n_experts < 1 || !q_a || !s_a || !nib_out || !scale_out) return MOE_EINVAL;
  const size_t H = (size_t)dims->hidden, I = (size_t)dims->inter;
  const size_t NB = H / 32, NBI = I / 32;
  if (which == MOE_GATEUP) {
    // [E][I][2: gate, up][H/32 blocks][16 B], scales [E][I][2][H/32]; block b of row
    // (i, m) at position block_pos(b, i)
    if (!q_b || !s_b) return MOE_EINVAL;
    for (size_t e = 0; e < (size_t)n_experts; ++e) {
      uint8_t* nib = nib_out + e * gu_nib_bytes(*dims);
      uint16_t* sc = scale_out + e * (gu_sc_bytes(*dims) / 2);
      for (size_t i = 0; i < I; ++i)
        for (size_t m = 0; m < 2; ++m) {
          const int8_t* q = (m == 0 ? q_a : q_b) + e * I * H + i * H;
          const uint16_t* sv = (m == 0 ? s_a : s_b) + e * I * NB + i * NB;
          const size_t base = (i * 2 + m) * NB;
          for (size_t b = 0; b < NB; ++b) {
            const size_t pb = (size_t)block_pos((int)b, (int)i);
            if (!pack_block(q + b * 32, nib + (base + pb) * 16)) return MOE_EINVAL;
            sc[base + pb] = sv[b];
          }
        }
    }
    return MOE_OK;
  }
  if (which == MOE_DOWN) {
    // block-major: codes [E][I/32 blocks][H rows][16 B], scales [E][I/32][H]; block b of
    // every output row of an expert is one contiguous run of H blocks
    for (size_t e = 0; e < (size_t)n_experts; ++e) {
      uint8_t* nib = nib_out + e * dn_nib_bytes(*dims);
      uint16_t* sc = scale_out + e * (dn_sc_bytes(*dims) / 2);
      const int8_t* q = q_a + e * H * I;
      const uint16_t* sv = s_a + e * H * NBI;
      for (size_t b = 0; b < NBI; ++b)
        for (size_t o = 0; o < H; ++o) {
          if (!pack_block(q + o * I + b * 32, nib + (b * H + o) * 16)) return MOE_EINVAL;
          sc[b * H + o] = sv[o * NBI + b];
        }
    }
    return MOE_OK;
  }
  return MOE_EINVAL;
}

int moe_round_host(moe_handle* h, const moe_dims* dims, const moe_layer_w* layers, int32_t L,
                   const uint16_t* x_host, int32_t rows, float* out_host, uint16_t* x_dev,
                   float* out_dev, int32_t* stats, void* ws, size_t ws_bytes, int use_graph, int sync,
                   void* stream) {
  // every argument check comes before the first copy is enqueued
  if (!h || !dims || !layers || !x_host || !out_host || !x_dev || !out_dev) return MOE_EINVAL;
  const int rc = check_dims(dims);
  if (rc != MOE_OK) return rc;
  if (L < 1 || L > kMaxLayers || rows < 1 || rows > dims->max_rows) return MOE_EINVAL;
  const size_t n = (size_t)L * (size_t)rows * (size_t)dims->hidden;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(x_dev, x_host, n * sizeof(uint16_t), cudaMemcpyHostToDevice, st) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ECUDA;
  }
  const int r = moe_round(h, layers, L, x_dev, rows, out_dev, stats, ws, ws_bytes, use_graph, stream);
  if (r != MOE_OK) return r;
  if (cudaMemcpyAsync(out_host, out_dev, n * sizeof(float), cudaMemcpyDeviceToHost, st) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ECUDA;
  }
  return sync ? moe_last_device_status(h, stream) : MOE_OK;
}

const char* moe_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_EINVAL: return "invalid argument (dimensions, NULL or misaligned pointer, rows)";
    case MOE_ECUDA: return "CUDA runtime error";
    case MOE_EWORKSPACE: return "workspace smaller than moe_workspace_bytes()";
    case MOE_ETIMEOUT: return "a bounded device-side wait gave up";
    case MOE_EUNSUPPORTED: return "dimensions outside what this build supports";
    default: return "unknown error code";
  }
}

}  // extern "C"
