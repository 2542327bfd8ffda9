// Host-side launch plans of the scan kernels (see cr_scan.cu).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "cr.h"
#include "cr_plan.h"

namespace cr {

struct ScanPlan {
  bool supported = false;
  int64_t batch = 0, n = 0;
  cr_policy policy = CR_LEFT_FOLD;
  int64_t B = 1;
  size_t ws_bytes = kHeaderBytes;
};

bool scan_args_ok(cr_policy p, int64_t B);
ScanPlan plan_scan(int64_t batch, int64_t n, cr_policy p, int64_t B, size_t esize);

template <class T>
cudaError_t run_scan(const ScanPlan& plan, const T* x, T* out, int64_t elem_stride,
                     int64_t batch_stride, char* ws, cudaStream_t s);

}  // namespace cr
