// Canonical scan kernels (placeholder: no policy implemented yet).
#include "cr_device.cuh"
#include "cr_scan.h"

namespace cr {

bool scan_args_ok(cr_policy p, int64_t B) {
  switch (p) {
    case CR_LEFT_FOLD:
    case CR_PAIRWISE:
    case CR_ITERATED_PAIRWISE: return true;
    case CR_BLOCK_DYADIC: return B >= 1 && (B & (B - 1)) == 0;
    default: return false;
  }
}

ScanPlan plan_scan(int64_t batch, int64_t n, cr_policy p, int64_t B, size_t) {
  ScanPlan plan;
  plan.batch = batch;
  plan.n = n;
  plan.policy = p;
  plan.B = B;
  plan.supported = false;
  return plan;
}

template <class T>
cudaError_t run_scan(const ScanPlan&, const T*, T*, int64_t, int64_t, char*, cudaStream_t) {
  return cudaErrorNotSupported;
}
template cudaError_t run_scan<double>(const ScanPlan&, const double*, double*, int64_t,
                                      int64_t, char*, cudaStream_t);
template cudaError_t run_scan<float>(const ScanPlan&, const float*, float*, int64_t, int64_t,
                                     char*, cudaStream_t);

}  // namespace cr
