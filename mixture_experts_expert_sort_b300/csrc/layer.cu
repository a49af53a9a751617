// The whole MoE expert layer, forward and backward, as one call each: the
// sequence of the kernels above over a caller-owned workspace.
//
// Forward ("Efficient MoE Training for Biological Foundation Models",
// §Challenge 1 and §Challenge 3):
//   route -> expert-sort plan -> permute -> FC1 grouped GEMM with the fused
//   scaled SwiGLU -> FC2 grouped GEMM -> combine.
// Backward (chain rule of the same steps):
//   permute dOut -> FC2 dgrad with the fused SwiGLU backward -> FC2 wgrad ->
//   FC1 dgrad -> FC1 wgrad -> un-permute dXp -> route backward.
// MXFP8 (§Challenge 2 and 3): the permute of x and of dOut is fused into
// their row- and column-wise quantisation, both weights are quantised once
// per forward in both directions (row-wise copies serve the dgrads), the FC1
// and FC2-dgrad epilogues emit their outputs already quantised, and every
// GEMM consumes operands whose 32-blocks run along its reduction dimension.
// No host synchronisation: every size that depends on the routing stays on
// the device; buffers are sized by the host bound R_max = T*k + E*(align-1)
// (rounded up to a multiple of 128 in MXFP8 mode).
#include "common.cuh"

namespace moe {
namespace layer {

enum Part {
  P_IDX = 0, P_W, P_COUNTS, P_OFFSETS, P_DEST, P_SRC, P_PLAN_WS, P_PROWS, P_XP, P_GU, P_H,
  P_Y2, P_DY2, P_DY1, P_DXP, P_DP,
  // MXFP8 mode only: data (q) and tiled scales (s), row-wise and column-wise.
  P_XQ_ROW, P_XS_ROW, P_XQ_COL, P_XS_COL,
  P_W1Q_ROW, P_W1S_ROW, P_W1Q_COL, P_W1S_COL,
  P_W2Q_ROW, P_W2S_ROW, P_W2Q_COL, P_W2S_COL,
  P_HQ_ROW, P_HS_ROW, P_HQ_COL, P_HS_COL,
  P_DY2Q_ROW, P_DY2S_ROW, P_DY2Q_COL, P_DY2S_COL,
  P_DY1Q_ROW, P_DY1S_ROW, P_DY1Q_COL, P_DY1S_COL,
  // MXFP8_ACT4 mode only: the row-wise MXFP4 copies of x (gathered) and H.
  P_X4Q, P_X4S, P_H4Q, P_H4S,
  P_COUNT
};
static_assert(P_XQ_ROW == MOE_PART_XQ_ROW && P_W1Q_ROW == MOE_PART_W1Q_ROW &&
                  P_HQ_ROW == MOE_PART_HQ_ROW && P_DY1S_COL == MOE_PART_DY1S_COL &&
                  P_X4Q == MOE_PART_X4Q_ROW && P_H4Q == MOE_PART_H4Q_ROW,
              "part ids match include/moe.h");

struct Layout {
  size_t off[P_COUNT];
  size_t bytes[P_COUNT];
  size_t total;
  long long rmax;
  int parts;
};

static size_t up256(size_t b) { return (b + 255) / 256 * 256; }

static bool is_mx(const moe_layer_config* c) {
  return c->precision == MOE_PRECISION_MXFP8 || c->precision == MOE_PRECISION_MXFP8_ACT4;
}
static bool is_act4(const moe_layer_config* c) { return c->precision == MOE_PRECISION_MXFP8_ACT4; }

static bool config_ok(const moe_layer_config* c) {
  if (!c) return false;
  if (c->T < 1 || c->H < 128 || c->H % 128 || c->F < 128 || c->F % 128 || c->E < 1 ||
      c->E > 256 || c->k < 1 || c->k > 8 || c->k > c->E)
    return false;
  if (c->align < 128 || c->align % 128 || c->align > 4096) return false;
  if (c->precision != MOE_PRECISION_BF16 && !is_mx(c)) return false;
  // MXFP8 wgrad tiles are 256 output columns wide: FC2's wgrad has N = H.
  if (is_mx(c) && c->H % 256) return false;
  long long rmax = (long long)c->T * c->k + (long long)c->E * (c->align - 1);
  if (is_mx(c)) rmax = (rmax + 127) / 128 * 128;
  if ((long long)c->E * c->H >= (1LL << 31) || (long long)c->E * c->F >= (1LL << 31)) return false;
  return rmax < (1LL << 31);
}

static size_t mx_scale_bytes(size_t mn, size_t kdim) { return (mn / 128) * (kdim / 128) * 512; }

static Layout layout(const moe_layer_config* c) {
  Layout L{};
  const long long Tk = (long long)c->T * c->k;
  const bool mx = is_mx(c);
  L.rmax = Tk + (long long)c->E * (c->align - 1);
  if (mx) L.rmax = (L.rmax + 127) / 128 * 128;
  L.parts = mx ? 2 * ((c->F + 255) / 256) : moe_swiglu_bwd_parts(c->F);
  const size_t R = (size_t)L.rmax, H = c->H, F = c->F, E = c->E;
  const size_t bf = mx ? 0 : 1;  // bf16 activations that MXFP8 mode keeps quantised instead
  const size_t q = mx ? 1 : 0;
  L.bytes[P_IDX] = Tk * 4;
  L.bytes[P_W] = Tk * 4;
  L.bytes[P_COUNTS] = (size_t)c->E * 4;
  L.bytes[P_OFFSETS] = (size_t)(c->E + 1) * 4;
  L.bytes[P_DEST] = Tk * 4;
  L.bytes[P_SRC] = R * 4;
  L.bytes[P_PLAN_WS] = moe_permute_plan_workspace_size(c->T, c->E, c->k);
  L.bytes[P_PROWS] = R * 4;
  L.bytes[P_XP] = bf * R * H * 2;
  L.bytes[P_GU] = R * 2 * F * 2;
  L.bytes[P_H] = bf * R * F * 2;
  L.bytes[P_Y2] = R * H * 2;
  L.bytes[P_DY2] = bf * R * H * 2;
  L.bytes[P_DY1] = bf * R * 2 * F * 2;
  L.bytes[P_DXP] = R * H * 2;
  L.bytes[P_DP] = R * (size_t)L.parts * 4;
  // MXFP8 operand pairs: (rows, cols) of the row-wise copy; the column-wise
  // copy is its transpose [cols, rows].
  const size_t mxdims[6][2] = {{R, H}, {E * H, 2 * F}, {E * F, H},
                               {R, F}, {R, H},         {R, 2 * F}};
  const int mxfirst[6] = {P_XQ_ROW, P_W1Q_ROW, P_W2Q_ROW, P_HQ_ROW, P_DY2Q_ROW, P_DY1Q_ROW};
  for (int i = 0; i < 6; ++i) {
    const size_t m = mxdims[i][0], n = mxdims[i][1];
    L.bytes[mxfirst[i] + 0] = q * m * n;
    L.bytes[mxfirst[i] + 1] = q * mx_scale_bytes(m, n);
    L.bytes[mxfirst[i] + 2] = q * m * n;
    L.bytes[mxfirst[i] + 3] = q * mx_scale_bytes(n, m);
  }
  const size_t a4 = is_act4(c) ? 1 : 0;
  L.bytes[P_X4Q] = a4 * R * H / 2;
  L.bytes[P_X4S] = a4 * mx_scale_bytes(R, H);
  L.bytes[P_H4Q] = a4 * R * F / 2;
  L.bytes[P_H4S] = a4 * mx_scale_bytes(R, F);
  // MXFP4-activation mode: x and H reach the backward only as their MXFP4
  // copies. Their row-wise FP8 copies are dead once the forward is done, so
  // the column-wise FP8 operands the backward rebuilds for the two wgrads
  // take the same bytes (a [cols, rows] copy has the size of its [rows, cols]
  // one, scales included), and the forward writes no column-wise H.
  auto aliased = [&](int i) {
    return a4 && (i == P_XQ_COL || i == P_XS_COL || i == P_HQ_COL || i == P_HS_COL);
  };
  size_t o = 0;
  for (int i = 0; i < P_COUNT; ++i) {
    if (aliased(i)) continue;
    L.off[i] = o;
    o += up256(L.bytes[i]);
  }
  if (a4) {
    L.off[P_XQ_COL] = L.off[P_XQ_ROW];
    L.off[P_XS_COL] = L.off[P_XS_ROW];
    L.off[P_HQ_COL] = L.off[P_HQ_ROW];
    L.off[P_HS_COL] = L.off[P_HS_ROW];
  }
  L.total = o;
  return L;
}

#define MOE_TRY(x)             \
  do {                         \
    int _s = (x);              \
    if (_s != MOE_OK) return _s; \
  } while (0)

}  // namespace layer
}  // namespace moe

using namespace moe::layer;

extern "C" size_t moe_layer_workspace_size(const moe_layer_config* cfg) {
  if (!config_ok(cfg)) return 0;
  return layout(cfg).total;
}

extern "C" int moe_layer_workspace_part(const moe_layer_config* cfg, int part, size_t* offset,
                                        size_t* bytes) {
  if (!config_ok(cfg) || part < 0 || part >= P_COUNT || !offset || !bytes) return MOE_ERR_ARG;
  Layout L = layout(cfg);
  *offset = L.off[part];
  *bytes = L.bytes[part];
  return MOE_OK;
}

extern "C" int moe_layer_forward(const moe_layer_config* cfg, const float* logits, const void* x,
                                 const void* w1, const void* w2, void* out, void* workspace,
                                 size_t workspace_bytes, moe_stream_t stream) {
  if (!config_ok(cfg) || !logits || !x || !w1 || !w2 || !out || !workspace) return MOE_ERR_ARG;
  Layout L = layout(cfg);
  if (workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MOE_ERR_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto P = [&](int i) { return ws + L.off[i]; };
  const int T = cfg->T, H = cfg->H, F = cfg->F, E = cfg->E, k = cfg->k;
  int32_t* idx = (int32_t*)P(P_IDX);
  float* w = (float*)P(P_W);
  int32_t* counts = (int32_t*)P(P_COUNTS);
  int32_t* offsets = (int32_t*)P(P_OFFSETS);
  int32_t* dest = (int32_t*)P(P_DEST);
  int32_t* src = (int32_t*)P(P_SRC);
  float* p_rows = (float*)P(P_PROWS);
  MOE_TRY(moe_route(logits, T, E, k, idx, w, stream));
  MOE_TRY(moe_permute_plan(idx, T, E, k, cfg->align, counts, offsets, dest, src, L.rmax,
                           P(P_PLAN_WS), L.bytes[P_PLAN_WS], stream));
  if (is_mx(cfg)) {
    const long long R = L.rmax;
    // per-row routing weights only; the gather of x is fused into its quantisation
    MOE_TRY(moe_permute(x, dest, offsets, counts, w, T, H, E, k, nullptr, p_rows, stream));
    // ACT4: the column-wise copy of x is rebuilt from MXFP4 in the backward
    MOE_TRY(mxfp8_quantize(x, R, H, H, src, k,
                           is_act4(cfg) ? MOE_QUANT_ROWWISE : MOE_QUANT_ROWWISE | MOE_QUANT_COLWISE,
                           P(P_XQ_ROW), P(P_XS_ROW), P(P_XQ_COL), P(P_XS_COL), stream));
    if (is_act4(cfg))
      MOE_TRY(mxfp4_from_mxfp8(P(P_XQ_ROW), P(P_XS_ROW), R, H, P(P_X4Q), P(P_X4S), stream));
    MOE_TRY(mxfp8_quantize(w1, (long long)E * H, 2 * F, 2 * F, nullptr, 1,
                           MOE_QUANT_ROWWISE | MOE_QUANT_COLWISE, P(P_W1Q_ROW), P(P_W1S_ROW),
                           P(P_W1Q_COL), P(P_W1S_COL), stream));
    MOE_TRY(mxfp8_quantize(w2, (long long)E * F, H, H, nullptr, 1,
                           MOE_QUANT_ROWWISE | MOE_QUANT_COLWISE, P(P_W2Q_ROW), P(P_W2S_ROW),
                           P(P_W2Q_COL), P(P_W2S_COL), stream));
    // ACT4: no column-wise H (its bytes are the row-wise H that FC2 reads)
    MOE_TRY(moe_fc1_swiglu_mxfp8(P(P_XQ_ROW), P(P_XS_ROW), R, H, P(P_W1Q_COL), P(P_W1S_COL),
                                 offsets, p_rows, E, F, P(P_GU), P(P_HQ_ROW), P(P_HS_ROW),
                                 is_act4(cfg) ? nullptr : P(P_HQ_COL),
                                 is_act4(cfg) ? nullptr : P(P_HS_COL), stream));
    if (is_act4(cfg))  // H is carried to the backward as MXFP4
      MOE_TRY(mxfp4_from_mxfp8(P(P_HQ_ROW), P(P_HS_ROW), R, F, P(P_H4Q), P(P_H4S), stream));
    // FC2: B_e[n, f] = W2_e[f, n] from the column-wise copy [H, E*F] (blocks along F)
    MOE_TRY(moe_grouped_gemm_mxfp8(MOE_GEMM_FPROP, P(P_HQ_ROW), P(P_HS_ROW), R, F, P(P_W2Q_COL),
                                   P(P_W2S_COL), H, (long long)E * F, 0, F, offsets, E, 0, H, F,
                                   P(P_Y2), stream));
    MOE_TRY(moe_unpermute(P(P_Y2), dest, nullptr, T, H, k, out, stream));
    return MOE_OK;
  }
  MOE_TRY(moe_permute(x, dest, offsets, counts, w, T, H, E, k, P(P_XP), p_rows, stream));
  MOE_TRY(moe_fc1_swiglu_bf16(P(P_XP), w1, offsets, p_rows, E, L.rmax, H, F, P(P_GU), P(P_H),
                              nullptr, stream));
  MOE_TRY(moe_grouped_gemm_bf16(MOE_GEMM_FPROP, P(P_H), w2, 0, offsets, E, L.rmax, 0, H, F,
                                P(P_Y2), nullptr, nullptr, stream));
  MOE_TRY(moe_unpermute(P(P_Y2), dest, nullptr, T, H, k, out, stream));
  return MOE_OK;
}

extern "C" int moe_layer_backward(const moe_layer_config* cfg, const void* dout, const void* w1,
                                  const void* w2, void* dx, void* dw1, void* dw2, float* dlogits,
                                  void* workspace, size_t workspace_bytes, moe_stream_t stream) {
  if (!config_ok(cfg) || !dout || !w1 || !w2 || !dx || !dw1 || !dw2 || !dlogits || !workspace)
    return MOE_ERR_ARG;
  Layout L = layout(cfg);
  if (workspace_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return MOE_ERR_ARG;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  auto P = [&](int i) { return ws + L.off[i]; };
  const int T = cfg->T, H = cfg->H, F = cfg->F, E = cfg->E, k = cfg->k;
  int32_t* idx = (int32_t*)P(P_IDX);
  float* w = (float*)P(P_W);
  int32_t* counts = (int32_t*)P(P_COUNTS);
  int32_t* offsets = (int32_t*)P(P_OFFSETS);
  int32_t* dest = (int32_t*)P(P_DEST);
  float* p_rows = (float*)P(P_PROWS);
  float* dp = (float*)P(P_DP);
  if (is_mx(cfg)) {
    const long long R = L.rmax;
    const int32_t* src = (const int32_t*)P(P_SRC);
    // permute of dOut fused into its row-wise (dgrad) and column-wise (wgrad) quantisation
    MOE_TRY(mxfp8_quantize(dout, R, H, H, src, k, MOE_QUANT_ROWWISE | MOE_QUANT_COLWISE,
                           P(P_DY2Q_ROW), P(P_DY2S_ROW), P(P_DY2Q_COL), P(P_DY2S_COL), stream));
    MOE_TRY(moe_fc2_dgrad_swiglu_bwd_mxfp8(P(P_DY2Q_ROW), P(P_DY2S_ROW), R, H, P(P_W2Q_ROW),
                                           P(P_W2S_ROW), offsets, p_rows, P(P_GU), E, F,
                                           P(P_DY1Q_ROW), P(P_DY1S_ROW), P(P_DY1Q_COL),
                                           P(P_DY1S_COL), dp, stream));
    // ACT4: the column-wise operands of the two wgrads come from the MXFP4
    // copies, into the bytes of the (now dead) row-wise FP8 copies
    if (is_act4(cfg)) {
      MOE_TRY(mxfp8_colwise_from_mxfp4_rowwise(P(P_H4Q), P(P_H4S), R, F, P(P_HQ_COL), P(P_HS_COL),
                                               stream));
      MOE_TRY(mxfp8_colwise_from_mxfp4_rowwise(P(P_X4Q), P(P_X4S), R, H, P(P_XQ_COL), P(P_XS_COL),
                                               stream));
    }
    // dW2_e = H_e^T dY2_e, both column-wise (blocks along the group's rows)
    MOE_TRY(moe_grouped_gemm_mxfp8(MOE_GEMM_WGRAD, P(P_HQ_COL), P(P_HS_COL), F, R, P(P_DY2Q_COL),
                                   P(P_DY2S_COL), H, R, 0, 0, offsets, E, F, H, 0, dw2, stream));
    // dXp = dY1 W1_e^T: B_e[n, c] = W1_e[n, c] from the row-wise copy [E*H, 2F]
    MOE_TRY(moe_grouped_gemm_mxfp8(MOE_GEMM_FPROP, P(P_DY1Q_ROW), P(P_DY1S_ROW), R, 2 * F,
                                   P(P_W1Q_ROW), P(P_W1S_ROW), (long long)E * H, 2 * F, H, 0,
                                   offsets, E, 0, H, 2 * F, P(P_DXP), stream));
    // dW1_e = Xp_e^T dY1_e
    MOE_TRY(moe_grouped_gemm_mxfp8(MOE_GEMM_WGRAD, P(P_XQ_COL), P(P_XS_COL), H, R, P(P_DY1Q_COL),
                                   P(P_DY1S_COL), 2 * F, R, 0, 0, offsets, E, H, 2 * F, 0, dw1,
                                   stream));
    MOE_TRY(moe_unpermute(P(P_DXP), dest, nullptr, T, H, k, dx, stream));
    MOE_TRY(moe_route_backward(dp, L.parts, L.parts, dest, w, idx, T, E, k, dlogits, stream));
    return MOE_OK;
  }
  MOE_TRY(moe_permute(dout, dest, offsets, counts, nullptr, T, H, E, k, P(P_DY2), nullptr, stream));
  MOE_TRY(moe_fc2_dgrad_swiglu_bwd_bf16(P(P_DY2), w2, offsets, p_rows, P(P_GU), E, L.rmax, H, F,
                                        P(P_DY1), dp, nullptr, stream));
  MOE_TRY(moe_grouped_gemm_bf16(MOE_GEMM_WGRAD, P(P_H), P(P_DY2), 0, offsets, E, L.rmax, F, H, 0,
                                dw2, nullptr, nullptr, stream));
  MOE_TRY(moe_grouped_gemm_bf16(MOE_GEMM_FPROP, P(P_DY1), w1, 1, offsets, E, L.rmax, 0, H, 2 * F,
                                P(P_DXP), nullptr, nullptr, stream));
  MOE_TRY(moe_grouped_gemm_bf16(MOE_GEMM_WGRAD, P(P_XP), P(P_DY1), 0, offsets, E, L.rmax, H,
                                2 * F, 0, dw1, nullptr, nullptr, stream));
  MOE_TRY(moe_unpermute(P(P_DXP), dest, nullptr, T, H, k, dx, stream));
  MOE_TRY(moe_route_backward(dp, L.parts, L.parts, dest, w, idx, T, E, k, dlogits, stream));
  return MOE_OK;
}
