// Launchers shared between the translation units of libf8 (host side only).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace f8 {

struct DeviceInfo {
    int ordinal = -1;
    int sm_count = 0;
    int cc_major = 0;
    int cc_minor = 0;
    unsigned *status = nullptr; // device address of this device's status word
};

// Per-device facts, filled on first use of a device (thread-safe).
// Returns nullptr if the device cannot be queried.
const DeviceInfo *device_info();

// Time limit of the GEMM pipeline's device waits.
uint64_t wait_limit_ns();

// amax over n bf16 values; n >= 1, x 16-byte aligned.
cudaError_t launch_amax(const void *x, int64_t n, float *amax_out, const DeviceInfo &dev,
                        cudaStream_t stream);

// Scale + cast + (optional) transpose of a [rows, cols] bf16 tensor.
cudaError_t launch_cast_transpose(const void *x, int64_t rows, int64_t cols, const float *amax,
                                  float *scale_out, uint8_t *q, uint8_t *q_t,
                                  const DeviceInfo &dev, cudaStream_t stream);

// C[M,N] = bf16(A[M,K] B[N,K]^T / (sa sb)); M, N, K >= 1, K % 16 == 0.
// Returns cudaErrorNotSupported if the tensor-map encoder is unavailable.
cudaError_t launch_gemm(const uint8_t *a, const uint8_t *b, int64_t M, int64_t N, int64_t K,
                        const float *sa, const float *sb, void *c, const DeviceInfo &dev,
                        cudaStream_t stream);

// One CTA waiting on an mbarrier that is never signalled (failure-path test).
cudaError_t launch_wait_selftest(uint64_t limit_ns, const DeviceInfo &dev, cudaStream_t stream);

} // namespace f8
