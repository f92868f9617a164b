// Definition of the opaque csa2_ctx (internal to the library).
#pragma once
#include <string>

#include "common.cuh"

struct csa2_ctx {
  csa2_config cfg;
  int device = 0;
  int num_sms = 0;
  csa2::RopeParams rope;
  uint32_t* d_flags = nullptr;
  unsigned long long* d_work = nullptr;  // [2] ticket counters of the index scan (zero between launches)
  cudaStream_t side = nullptr;    // step side stream: compress and the tail scores, then the window tile
  cudaEvent_t ev_fork = nullptr;  // recorded on the caller's stream at the start of a step
  cudaEvent_t ev_idx = nullptr;   // recorded on the caller's stream after the index scan
  cudaEvent_t ev_tail = nullptr;  // recorded on the side stream after compress and the tail scores
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
