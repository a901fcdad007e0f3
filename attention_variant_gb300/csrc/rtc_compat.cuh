// rtc_compat.cuh -- the few host-header types the kernel sources use, for
// both compilers that build them: nvcc (the library) and the runtime compiler
// NVRTC (kernels specialised for a score_mod expression at run time), which
// has no host headers.
#pragma once

#ifdef __CUDACC_RTC__
typedef unsigned char uint8_t;
typedef unsigned short uint16_t;
typedef unsigned int uint32_t;
typedef unsigned long long uint64_t;
typedef signed char int8_t;
typedef short int16_t;
typedef int int32_t;
typedef long long int64_t;
// The driver's opaque 128-byte, 64-byte-aligned tensor-map type.
struct alignas(64) CUtensorMap_st {
    unsigned long long opaque[16];
};
typedef CUtensorMap_st CUtensorMap;
#else
#include <cstdint>
#include <cuda.h>
#endif
