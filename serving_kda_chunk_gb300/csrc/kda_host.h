// kda_host.h -- host-side argument checks shared by the libkda entry points.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool dtype_ok(kda_dtype d) { return d == KDA_BF16 || d == KDA_F32; }

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

// Map the last launch error to a status (clears the sticky-free error state).
inline kda_status launch_status() {
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // namespace kda

#define KDA_REQUIRE(cond, code) \
    do {                        \
        if (!(cond)) return (code); \
    } while (0)
