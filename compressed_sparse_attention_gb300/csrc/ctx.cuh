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
  std::string err;
  int last_launches = 0;
};
