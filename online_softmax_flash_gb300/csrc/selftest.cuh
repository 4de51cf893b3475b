// Self-test of the bounded device waits (osf_selftest_bounded_wait).
#pragma once
#include "osf_internal.cuh"

namespace osf {
cudaError_t launch_bounded_wait_selftest(unsigned long long limit_ns, int *status, cudaStream_t s);
}  // namespace osf
