// Definition of the opaque csa2_ctx (internal to the library).
#pragma once
#include <string>

#include "common.cuh"

struct csa2_ctx {
  csa2_config cfg;
  int device = 0;
  int num_sms = 0;
  int prio_high = 0;  // the device's greatest stream priority: the side stream's, and the window tile's launches
  csa2::RopeParams rope;
  uint32_t* d_flags = nullptr;
  unsigned long long* d_work = nullptr;  // [2] ticket counters of the index scan (zero between launches)
  cudaStream_t side = nullptr;    // step side stream: a candidate source's pool, beside its attention
  cudaEvent_t ev_join = nullptr;  // recorded on the side stream after its last launch
  cudaEvent_t ev_topk = nullptr;  // recorded on the caller's stream after a candidate source's top-k
  cudaStream_t copy = nullptr;    // host-buffer steps: the copy of q beside the first half of the step
  cudaEvent_t ev_copy = nullptr;  // recorded on the caller's stream before that copy
  cudaEvent_t ev_q = nullptr;     // recorded on the copy stream once q is on the device
  // csa2_attend_noalloc: device address of the library's fixed scratch array on
  // this context's device, looked up by the first such call on this context
  void* noalloc_scratch = nullptr;
  std::string err;
  int last_launches = 0;
};
