// Host-side state of a moe_plan (shared by the C-ABI translation units).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"

typedef CUresult (*encode_tiled_fn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

namespace moe {
// A forward's routing and schedule inside its workspace (device pointers)
struct FwdRoutingViews {
  const int* topk_idx;
  const float* topk_w;
  const float* topk_logit;
  const int* M;
  const int* S;
  const int* sched;
};
int fwd_routing_views(const moe_plan* pl, int64_t T, const void* workspace, FwdRoutingViews* v);
}  // namespace moe

struct moe_plan {
  moe_config cfg;
  int device;
  int num_sms;
  int grid;  // persistent kernel CTAs = gather + gemm
  encode_tiled_fn encode;
  cudaEvent_t timing[4];  // optional, see moe_plan_set_timing_events
  bool timed;
  cudaEvent_t bwd_timing[5];  // optional, see moe_plan_set_bwd_timing_events
  bool bwd_timed;
};
