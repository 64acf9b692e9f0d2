// a5-a7: routed MoE layer with int4g experts (route, permute, grouped
// gate/up + SwiGLU, grouped down + weighted combine).
#include "fl_common.cuh"

extern "C" int fl_moe_int4g_workspace(int M, int E, int k, int H, int I, int has_shared, size_t* out) {
  (void)M; (void)E; (void)k; (void)H; (void)I; (void)has_shared; (void)out;
  return FL_ERR_UNSUPPORTED;
}

extern "C" int fl_moe_int4g(const void* x, const float* logits, int M, int H, int E, int k, int I, int scoring,
                            int renorm, const void* w13, const void* w2, const void* shared_w13,
                            const void* shared_w2, void* y, int32_t* topk_ids, float* topk_w,
                            int32_t* expert_offsets, int32_t* perm, void* ws, size_t ws_bytes,
                            fl_stream_t stream) {
  return FL_ERR_UNSUPPORTED;
}
