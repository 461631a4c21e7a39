// halo_noalloc.cu -- a coordinate exchange that allocates no device memory.
//
// halo_exchange_x_noalloc runs the same fused coordinate kernel as
// halo_exchange_x, but takes its scratch -- the per-(domain, pulse) arrival
// counters and the work ticket -- from a fixed array compiled into this
// library instead of from memory the plan allocated.  It is meant for callers
// that may not allocate device memory when they call in: code running inside
// a host framework whose pool allocator owns all device memory and forbids
// allocations behind its back, and latency-critical loops in which a
// cudaMalloc / cudaFree (each of which can synchronise the whole device)
// is not acceptable.  The call itself makes no cudaMalloc, cudaFree or other
// allocating call; it needs a plan built earlier with halo_setup.
//
// The array is shared by every call on a device and keeps the last call's
// contents, so each call first clears the part it uses.  Calls whose kernels
// overlap on the GPU (different streams, or different host threads) race on
// the array and give wrong results.  The array holds kNoAllocMaxCounters
// counters: plans with n_domains * n_pulses above that are rejected with
// HALO_ESCRATCH.  Every GPU that loads the library holds the array (64 KiB)
// until the process exits.
//
// Where the array lives: halo_setup (which allocates anyway) looks up the
// array's device address once per device, with that device current.  Under
// lazy module loading that lookup is what places the array in device
// memory, so the no-allocation call itself only reads the stored address.
#include <atomic>
#include <mutex>

#include "halo_internal.cuh"

namespace {

constexpr int kNoAllocMaxCounters = HALO_NOALLOC_MAX_COUNTERS;
constexpr size_t kTicketBytes = 256;  // the ticket (8 bytes) in its own 256-byte block
constexpr size_t kScratchBytes = kTicketBytes + sizeof(uint32_t) * kNoAllocMaxCounters;

// [0, 8): work ticket (u64); [256, 256 + 4 * kNoAllocMaxCounters): arrival counters
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
std::atomic<void*> g_scratch_addr[kMaxDevices] = {};

}  // namespace

namespace halo {

// Device address of the array on the current device.  In host code the
// array's name only stands in for the symbol, so the address is looked up
// (once per device, with that device current) and stored.
int noalloc_prepare() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return HALO_ECUDA;
    if (dev >= kMaxDevices) return HALO_OK;  // no fixed array there: the call reports HALO_ECUDA
    std::lock_guard<std::mutex> guard(g_lock);
    if (!g_scratch_addr[dev].load()) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            (void)cudaGetLastError();
            return HALO_ECUDA;
        }
        g_scratch_addr[dev].store(p);
    }
    return HALO_OK;
}

}  // namespace halo

namespace {

// The stored address for the plan's device (set by halo_setup), or null.
void* scratch_address(int dev) {
    return dev >= 0 && dev < kMaxDevices ? g_scratch_addr[dev].load() : nullptr;
}

}  // namespace

extern "C" int halo_exchange_x_noalloc(halo_plan* pl, float* local_coords, void* stream) {
    if (!pl || !local_coords || ((uintptr_t)local_coords & 3u) || !pl->valid || !pl->fused_ready)
        return HALO_EINVAL;
    const int64_t counters = (int64_t)pl->n_dom * pl->P;
    if (counters > kNoAllocMaxCounters) return HALO_ESCRATCH;
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return HALO_ECUDA;
    if (prev != pl->dev && cudaSetDevice(pl->dev) != cudaSuccess) return HALO_ECUDA;
    int rc = HALO_OK;
    void* base = nullptr;
    const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    base = scratch_address(pl->dev);
    if (!base) rc = HALO_ECUDA;
    if (rc == HALO_OK && pl->n_items_x > 0) {
        // clear the ticket block and the counters this plan uses
        const size_t bytes = kTicketBytes + sizeof(uint32_t) * (size_t)counters;
        rc = halo::cuda_code(cudaMemsetAsync(base, 0, bytes, st));
        if (rc == HALO_OK)
            rc = halo::launch_exchange_x_scratch(
                pl, local_coords,
                reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(base) + kTicketBytes),
                reinterpret_cast<unsigned long long*>(base), st);
    }
    if (prev != pl->dev) cudaSetDevice(prev);
    return rc;
}
