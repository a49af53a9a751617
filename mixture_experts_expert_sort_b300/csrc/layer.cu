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
// No host synchronisation: every size that depends on the routing stays on
// the device; buffers are sized by the host bound R_max = T*k + E*(align-1).
#include "common.cuh"

namespace moe {
namespace layer {

enum Part {
  P_IDX = 0, P_W, P_COUNTS, P_OFFSETS, P_DEST, P_SRC, P_PLAN_WS, P_PROWS, P_XP, P_GU, P_H,
  P_Y2, P_DY2, P_DY1, P_DXP, P_DP, P_COUNT
};

struct Layout {
  size_t off[P_COUNT];
  size_t bytes[P_COUNT];
  size_t total;
  long long rmax;
  int parts;
};

static size_t up256(size_t b) { return (b + 255) / 256 * 256; }

static bool config_ok(const moe_layer_config* c) {
  if (!c) return false;
  if (c->T < 1 || c->H < 128 || c->H % 128 || c->F < 128 || c->F % 128 || c->E < 1 ||
      c->E > 256 || c->k < 1 || c->k > 8 || c->k > c->E)
    return false;
  if (c->align < 128 || c->align % 128 || c->align > 4096) return false;
  if (c->precision != MOE_PRECISION_BF16) return false;
  long long rmax = (long long)c->T * c->k + (long long)c->E * (c->align - 1);
  return rmax < (1LL << 31);
}

static Layout layout(const moe_layer_config* c) {
  Layout L{};
  const long long Tk = (long long)c->T * c->k;
  L.rmax = Tk + (long long)c->E * (c->align - 1);
  L.parts = moe_swiglu_bwd_parts(c->F);
  const size_t R = (size_t)L.rmax, H = c->H, F = c->F;
  L.bytes[P_IDX] = Tk * 4;
  L.bytes[P_W] = Tk * 4;
  L.bytes[P_COUNTS] = (size_t)c->E * 4;
  L.bytes[P_OFFSETS] = (size_t)(c->E + 1) * 4;
  L.bytes[P_DEST] = Tk * 4;
  L.bytes[P_SRC] = R * 4;
  L.bytes[P_PLAN_WS] = moe_permute_plan_workspace_size(c->T, c->E, c->k);
  L.bytes[P_PROWS] = R * 4;
  L.bytes[P_XP] = R * H * 2;
  L.bytes[P_GU] = R * 2 * F * 2;
  L.bytes[P_H] = R * F * 2;
  L.bytes[P_Y2] = R * H * 2;
  L.bytes[P_DY2] = R * H * 2;
  L.bytes[P_DY1] = R * 2 * F * 2;
  L.bytes[P_DXP] = R * H * 2;
  L.bytes[P_DP] = R * (size_t)L.parts * 4;
  size_t o = 0;
  for (int i = 0; i < P_COUNT; ++i) {
    L.off[i] = o;
    o += up256(L.bytes[i]);
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
  MOE_TRY(moe_permute(x, dest, offsets, counts, w, T, H, E, k, P(P_XP), p_rows, stream));
  MOE_TRY(moe_fc1_swiglu_bf16(P(P_XP), w1, offsets, p_rows, E, L.rmax, H, F, P(P_GU), P(P_H),
                              stream));
  MOE_TRY(moe_grouped_gemm_bf16(MOE_GEMM_FPROP, P(P_H), w2, 0, offsets, E, L.rmax, 0, H, F,
                                P(P_Y2), stream));
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
  MOE_TRY(moe_permute(dout, dest, offsets, counts, nullptr, T, H, E, k, P(P_DY2), nullptr, stream));
  MOE_TRY(moe_fc2_dgrad_swiglu_bwd_bf16(P(P_DY2), w2, offsets, p_rows, P(P_GU), E, L.rmax, H, F,
                                        P(P_DY1), dp, stream));
  MOE_TRY(moe_grouped_gemm_bf16(MOE_GEMM_WGRAD, P(P_H), P(P_DY2), 0, offsets, E, L.rmax, F, H, 0,
                                dw2, stream));
  MOE_TRY(moe_grouped_gemm_bf16(MOE_GEMM_FPROP, P(P_DY1), w1, 1, offsets, E, L.rmax, 0, H, 2 * F,
                                P(P_DXP), stream));
  MOE_TRY(moe_grouped_gemm_bf16(MOE_GEMM_WGRAD, P(P_XP), P(P_DY1), 0, offsets, E, L.rmax, H,
                                2 * F, 0, dw1, stream));
  MOE_TRY(moe_unpermute(P(P_DXP), dest, nullptr, T, H, k, dx, stream));
  MOE_TRY(moe_route_backward(dp, L.parts, L.parts, dest, w, idx, T, E, k, dlogits, stream));
  return MOE_OK;
}
