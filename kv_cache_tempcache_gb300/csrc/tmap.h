// TMA tensor maps and device facts used by the tensor-core kernels' launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fastar {

// A 3-D bf16 tensor map (d0 innermost, element units) with 128-byte swizzle and a
// box of box0 x box1 x box2; out-of-range elements read as zero.  Strides in bytes
// (multiples of 16).  Returns false if the driver rejects it.
bool make_tmap_bf16_3d(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                       uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1,
                       uint32_t box2 = 1);

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Opts kernel `func` into `bytes` of dynamic shared memory on the current device.  The
// attribute belongs to the device's context, so it is set once per (kernel, device)
// and remembered; returns the CUDA error of the first failed attempt.
cudaError_t opt_in_smem(const void* func, int bytes);

}  // namespace fastar
