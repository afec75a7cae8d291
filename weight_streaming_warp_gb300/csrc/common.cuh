// common.cuh -- device helpers and host-side launch plumbing shared by the kernels
// of libwsw.so (sm_103a only).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "wsw.h"

#define WSW_FULL_MASK 0xffffffffu

namespace wsw {

// ------------------------------------------------------------------ device --

// Programmatic dependent launch.  wait: block until every prerequisite grid has
// completed and its memory is visible (returns at once when the kernel was not
// launched with a programmatic dependency).  launch_dependents: allow the next
// kernel in the stream to be scheduled before this one finishes.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// L2 eviction policy for data that is read exactly once (streamed weights).
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Streaming loads of read-only data: not allocated in L1, evict-first in L2.
template <int BYTES>
struct StreamLoad;

template <>
struct StreamLoad<32> {
    __device__ __forceinline__ static void run(const void *p, uint32_t *v, uint64_t pol) {
        asm volatile(
            "ld.global.nc.L1::no_allocate.L2::cache_hint.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8], %9;"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
              "=r"(v[7])
            : "l"(p), "l"(pol));
    }
};

template <>
struct StreamLoad<16> {
    __device__ __forceinline__ static void run(const void *p, uint32_t *v, uint64_t pol) {
        asm volatile(
            "ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
            : "l"(p), "l"(pol));
    }
};
template <>
struct StreamLoad<8> {
    __device__ __forceinline__ static void run(const void *p, uint32_t *v, uint64_t pol) {
        asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0,%1}, [%2], %3;"
                     : "=r"(v[0]), "=r"(v[1])
                     : "l"(p), "l"(pol));
    }
};
template <>
struct StreamLoad<4> {
    __device__ __forceinline__ static void run(const void *p, uint32_t *v, uint64_t pol) {
        asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;"
                     : "=r"(v[0])
                     : "l"(p), "l"(pol));
    }
};
template <>
struct StreamLoad<2> {
    __device__ __forceinline__ static void run(const void *p, uint32_t *v, uint64_t pol) {
        unsigned short h;
        asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u16 %0, [%1], %2;"
                     : "=h"(h)
                     : "l"(p), "l"(pol));
        v[0] = h;
    }
};

// Load 16 bytes of streamed data at p (16-byte aligned when LB == 16) as LB-byte
// pieces.  The four 32-bit words come out identical whatever LB is.
template <int LB>
__device__ __forceinline__ void load16(const void *p, uint32_t (&v)[4], uint64_t pol) {
    const char *c = static_cast<const char *>(p);
    if constexpr (LB == 16) {
        StreamLoad<16>::run(c, v, pol);
    } else if constexpr (LB == 8) {
        StreamLoad<8>::run(c, v, pol);
        StreamLoad<8>::run(c + 8, v + 2, pol);
    } else if constexpr (LB == 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) StreamLoad<4>::run(c + 4 * i, v + i, pol);
    } else {
        static_assert(LB == 2, "load width");
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t lo, hi;
            StreamLoad<2>::run(c + 4 * i, &lo, pol);
            StreamLoad<2>::run(c + 4 * i + 2, &hi, pol);
            v[i] = lo | (hi << 16);
        }
    }
}

// Load 32 bytes of streamed data at p (32-byte aligned when LB == 32) as LB-byte
// pieces; the eight words come out identical whatever LB is.
template <int LB>
__device__ __forceinline__ void load32(const void *p, uint32_t (&v)[8], uint64_t pol) {
    if constexpr (LB == 32) {
        StreamLoad<32>::run(p, v, pol);
    } else {
        const char *c = static_cast<const char *>(p);
        uint32_t lo[4], hi[4];
        load16<(LB > 16 ? 16 : LB)>(c, lo, pol);
        load16<(LB > 16 ? 16 : LB)>(c + 16, hi, pol);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[i] = lo[i];
            v[4 + i] = hi[i];
        }
    }
}

__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// The CTA's threads request the 128-byte lines of [p, p + bytes) into L2, one line each.
__device__ __forceinline__ void prefetch_range_l2(const void *p, int64_t bytes) {
    const uintptr_t first = reinterpret_cast<uintptr_t>(p) & ~static_cast<uintptr_t>(127);
    const uintptr_t end = reinterpret_cast<uintptr_t>(p) + static_cast<uintptr_t>(bytes);
    for (uintptr_t l = first + 128 * static_cast<uintptr_t>(threadIdx.x); l < end; l += 128 * blockDim.x)
        prefetch_l2(reinterpret_cast<const void *>(l));
}

// bf16 pair in one 32-bit word -> two fp32 values (exact).
__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// ------------------------------------------------------------------- host --

struct DeviceInfo {
    int device;
    int sm_count;
    int max_smem_optin;
    int l2_bytes;
};

// Per-device properties, cached after the first query.  Returns false when the
// current device cannot be queried or is not an sm_103 part.
bool device_info(DeviceInfo *out, int *status);

// Resolve user launch options (NULL -> defaults).
struct Opts {
    int rows_per_warp;
    int load_bytes;
    bool pdl;
    int ctas_per_sm;
    int l2_prefetch_steps;  // resolved: 0 = off
};
int resolve_opts(const wsw_launch_opts *o, Opts *out);

// The widest load width (32, 16, 8, 4 or 2 bytes) that divides both the base
// address and the row pitch in bytes, capped at `cap`.
int load_width(const void *base, int64_t pitch_bytes, int cap);

// Raise a kernel's dynamic shared-memory limit to `bytes` once per device (later
// calls return without touching the driver, so they are safe during stream capture).
cudaError_t ensure_smem(const void *kernel, int bytes);

// Launch with optional programmatic stream serialization.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                   cudaStream_t stream, bool pdl, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace wsw
