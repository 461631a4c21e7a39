// halo_device.cuh -- device helpers shared by the exchange kernels.
#pragma once

#include <stdint.h>

#include "halo.h"

namespace halo {

// Debug builds (-DHALO_DEBUG): every slot index that a kernel gathers from or
// scatters to is checked against its buffer before the access; a bad one
// records HALO_EBOUNDS in the plan's error word (halo_status reports it) and
// the access is skipped.  Release builds compile the check away.
#ifdef HALO_DEBUG
__device__ __forceinline__ bool in_range(int64_t i, int64_t n, int* err) {
    if ((uint64_t)i < (uint64_t)n) return true;
    atomicCAS(err, 0, HALO_EBOUNDS);
    return false;
}
#else
__device__ __forceinline__ bool in_range(int64_t, int64_t, int*) { return true; }
#endif

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Exclusive scan across a block of NT threads (NT a multiple of 32, <= 1024).
template <int NT>
__device__ __forceinline__ int64_t block_exclusive_scan(int64_t v, int64_t* total) {
    __shared__ int64_t ws[NT / 32];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int64_t y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) ws[w] = x;
    __syncthreads();
    if (w == 0) {
        int64_t t = lane < NT / 32 ? ws[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int64_t y = __shfl_up_sync(kFull, t, o);
            if (lane >= o) t += y;
        }
        if (lane < NT / 32) ws[lane] = t;
    }
    __syncthreads();
    int64_t pre = (w > 0 ? ws[w - 1] : 0) + x - v;
    *total = ws[NT / 32 - 1];
    __syncthreads();
    return pre;
}


// A block's chunk of halo coordinates is one contiguous range of 12-byte
// slots in the destination domain.  The block stages it in shared memory and
// one thread writes it back with a bulk asynchronous copy (cp.async.bulk,
// shared -> global), which needs 16-byte aligned addresses and a multiple of
// 16 bytes: the 16-byte aligned middle goes by bulk copy, the at most three
// leading and three trailing floats by ordinary stores.
//
// Staging convention: the float that belongs at gdst[j] sits at
// stage[stage_shift(gdst) + j], so that global and shared addresses agree
// modulo 16.
__device__ __forceinline__ int stage_shift(const float* gdst) {
    return (int)(((uintptr_t)gdst & 15u) >> 2);
}

// Make this thread's generic-proxy writes to shared memory visible to the
// asynchronous proxy (every writing thread, before the block barrier).
__device__ __forceinline__ void fence_smem_to_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Called by one thread after the (warp or block) barrier.  complete = true:
// returns once the data is in global memory and ordered before this thread's
// later (release) operations; false: returns once the shared source has been
// read (enough before the block exits: kernel completion makes it visible).
__device__ __forceinline__ void bulk_store_floats(float* gdst, const float* stage, int nfloats,
                                                  bool complete) {
    const uintptr_t B = (uintptr_t)gdst;
    const int a = stage_shift(gdst);
    const uintptr_t Bend = B + 4 * (uintptr_t)nfloats;
    const uintptr_t Bup = (B + 15) & ~(uintptr_t)15;
    const uintptr_t Bdn = Bend & ~(uintptr_t)15;
    if (Bdn > Bup) {
        uint64_t g;
        asm("cvta.to.global.u64 %0, %1;" : "=l"(g) : "l"((uint64_t)Bup));
        const uint32_t s = (uint32_t)__cvta_generic_to_shared(stage + a) + (uint32_t)(Bup - B);
        const uint32_t size = (uint32_t)(Bdn - Bup);
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(g), "r"(s),
                     "r"(size)
                     : "memory");
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        for (uintptr_t x = B; x < Bup; x += 4) gdst[(x - B) >> 2] = stage[a + ((x - B) >> 2)];
        for (uintptr_t x = Bdn; x < Bend; x += 4) gdst[(x - B) >> 2] = stage[a + ((x - B) >> 2)];
        if (complete) {
            asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
            asm volatile("fence.proxy.async.global;" ::: "memory");
        } else {
            asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        }
    } else {
        for (int j = 0; j < nfloats; j++) gdst[j] = stage[a + j];
    }
}

// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may start while the kernel before it in the stream is still
// running; it reads only the plan's own tables (written by a rebuild, which
// ends with a synchronisation) before grid_dependency_wait(), which returns
// once the preceding grids have completed and their writes are visible.
// Every read of coordinates or forces, and every write, comes after it.
// Without the launch attribute both are no-ops.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next programmatically serialised kernel in the stream be scheduled
// as soon as every block of this one has started (its blocks still wait for
// this grid's completion before touching its data).
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace halo
