// halo_internal.cuh -- plan structure and the internal entry points shared by
// the translation units of libhalo.so.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "halo.h"

namespace halo {

constexpr int kThreads = 256;          // threads per block of every kernel here
constexpr int kHistTile = 1024;        // atoms per warp tile of the home partition
constexpr int kScanTile = 2048;        // elements per block of the device scan
constexpr int kMaxShards = HALO_MAX_SHARDS;

// Sharded data plane: shard k holds the dense slots [first[k], first[k + 1])
// in its own buffer ptr[k] (the domains of one z-slab), so dense slot g of
// shard k lives at ptr[k] + 3 * (g - first[k]).
struct ShardTable {
    float* ptr[kMaxShards];
    int64_t first[kMaxShards];
};

// Per (sender s, pulse p) description (host side, and the build-time kernels).
struct SPDesc {
    int64_t map_off;   // first entry of the index map in the plan's map array
    int64_t src_base;  // base[s]: first dense slot of the sender
    int64_t dst;       // base[r] + atomOffset: first dense slot of the halo slice in r
    int32_t send;      // entries
    int32_t split;     // entries below depOffset
    int32_t s, r, p, pad;
    float shift[3];
    float pad2;
};

// One chunk of coordinate work: entries [start, start+len) of one (s, p) map,
// all independent (below depOffset) or all dependent.  Self-contained, so a
// block needs one descriptor load per item.
struct XItem {
    int64_t map_off;     // index of the chunk's first map entry
    int64_t src_base;    // dense slot of the sender's local index 0
    int64_t dst;         // dense slot written by the chunk's first entry
    int32_t len;
    int32_t flag;        // counter released when done: arrived[r*P + p]
    int32_t wait_base;   // s*P: counters of the slices s received
    int16_t src_shard;   // shard of s (the sender) and of r (the receiver)
    int16_t dst_shard;
    uint64_t wait_mask;  // pulses q < p whose slices into s the entries reference
    float shift[3];
    int32_t pad2;
};

// One chunk of force work: pairs [off, off+len) of the reordered (src, dst)
// list; independent chunks wait for nothing.
struct FItem {
    int64_t off;
    int32_t len;
    int32_t flag;        // done[s*P + p]
    int32_t s_base;      // s*P
    int32_t r_base;      // r*P
    uint64_t ms, mr;     // later pulses to wait for, on s and on r (0 for independent)
    int16_t s_shard;     // shard of s (destination slots) and of r (halo sources)
    int16_t r_shard;
    int32_t pad;
};

}  // namespace halo

struct halo_plan {
    int dev = 0;
    int num_sms = 0;
    bool valid = false;              // false while (or after a failed) rebuild: exchanges refuse
    int grid[3] = {1, 1, 1};
    float box[3] = {0, 0, 0};
    float rc = 0;
    int n_dom = 0;
    int P = 0;
    int pulses_per_dim[3] = {0, 0, 0};
    int pulse_dim[HALO_MAX_PULSES] = {};
    int pulse_k[HALO_MAX_PULSES] = {};
    int64_t n_atoms = 0;
    int64_t n_local_total = 0;
    int64_t n_halo_total = 0;

    // host copies of the plan (filled after each build)
    std::vector<int32_t> n_home, n_local, send, split, own_off;  // own_off: n_dom*(P+1)
    std::vector<int64_t> base, map_off;                           // map_off: n_dom*P
    std::vector<halo::SPDesc> sp;

    // device memory owned by the plan: build
    float* d_bxyz = nullptr;        // build buffer (float4 per slot: x, y, z, forwarding dims):
                                    // home-compact region + halo regions
    int64_t cap_slots = 0;          // capacity of d_bxyz in slots (and of d_maps)
    int32_t* d_maps = nullptr;      // index maps, (pulse, sender) order
    int32_t* d_home_gid = nullptr;  // global id of each home-compact slot
    int64_t n_alloc_atoms = 0;
    int32_t* d_counts = nullptr;    // home partition tile counts (and scan output)
    int64_t counts_cap = 0;
    int32_t* d_scan_tmp = nullptr;
    int64_t scan_tmp_cap = 0;
    void* d_meta = nullptr;         // packed per-domain / per-pulse metadata (see build)
    size_t meta_bytes = 0;
    int32_t* d_pulse_scratch = nullptr;  // per-pulse block counts (3 * n_dom * B)
    int build_blocks_per_domain = 1;
    float* d_thr = nullptr;         // thresholds per pulse and sender cell
    int64_t debug_capacity = 0;     // test hook: build-buffer slots of the next build's first attempt
    int build_attempts = 0;         // attempts the last build needed (capacity retries + 1)
    uint32_t flags = 0;             // HALO_SETUP_* options
    double* d_faces = nullptr;      // corner pruning: lower faces [3][nmax], upper faces [3][nmax]

    // device memory owned by the plan: exchange
    halo::SPDesc* d_sp = nullptr;
    halo::XItem* d_items_x = nullptr;
    halo::FItem* d_items_f = nullptr;
    int64_t cap_sp = 0, cap_items_x = 0, cap_items_f = 0, cap_target = 0, cap_flags = 0,
            cap_nindep = 0;
    uint64_t* d_recv_mask = nullptr;  // per domain: pulses that delivered a nonempty slice
    int32_t* d_itemgen = nullptr;     // scratch of the device-side work-list generation
    int64_t cap_recv_mask = 0, cap_itemgen = 0;
    int n_items_x = 0, n_items_f = 0;
    std::vector<int32_t> max_chunks;  // per pulse: most chunks of one sender (utility grids)
    int chunk = 256;                // entries per work item
    int entries_per_thread = 1;
    int2* d_fpairs = nullptr;        // (src dense slot, dst dense slot) per force entry
    int64_t fpairs_cap = 0;
    int8_t* d_wmax = nullptr;        // last pulse adding into each dense slot (build time)
    int64_t wmax_cap = 0;
    int32_t* d_nindep = nullptr;     // independent force entries of each (s, p)
    uint32_t* d_target = nullptr;    // chunks per counter: arrived[n_dom*P] | done[n_dom*P]
    uint32_t* d_flags = nullptr;     // arrived[n_dom*P] | done[n_dom*P]
    unsigned long long* d_tickets = nullptr;  // [0] x, [1] f
    int* d_err = nullptr;            // sticky error word + where a wait gave up
    int grid_x = 0, grid_f = 0;
    long long wait_timeout_ns = 1000000000LL;
    int drop_flag = -1;              // test hook: arrived counter whose release is skipped
    unsigned long long* trace = nullptr;  // caller's trace buffer (device), or null
    int64_t trace_cap = 0;                // its size in items
    int64_t launches_x = 0, launches_f = 0;

    // pinned host staging for the build's host<->device copies (grow-only)
    void* h_stage = nullptr;
    size_t h_stage_cap = 0;
    void* h_stage_dev = nullptr;     // its device address (mapped), or null: copied with the copy engine
    bool stage_copies = false;       // never map the staging (HALO_STAGE_COPIES at setup)
    int occ_x = 0, occ_f = 0;        // resident blocks per SM of the fused kernels (cached)

    // sharded data plane: shard k holds the domains [shard_dom[k], shard_dom[k + 1])
    // (a z-slab of the grid) and the dense slots [shard_first[k], shard_first[k + 1])
    int n_shards = 1;
    bool shard_lists = false;        // halo_shard was called: rebuilds keep the FUSED work lists
    bool flat_chains_ready = false;  // the FLAT forwarding chains of this build are launched
    int home_grid_x = 1;             // blocks per domain of the home load / store kernels
    int shard_dom[halo::kMaxShards + 1] = {};
    int64_t shard_first[halo::kMaxShards + 1] = {};

    // exchange mode (HALO_MODE_*) and the flattened exchange's tables
    int mode = 0;
    bool fused_ready = false;        // FUSED work lists built for the current plan
    bool flat_ready = false;
    int32_t* d_xflat = nullptr;      // per halo slot: owner dense slot | shift bits << 29
    int4* d_xflat_items = nullptr;   // {flat halo index, dense slot, len, 0} per chunk
    int n_xflat_items = 0;
    int32_t* d_fown = nullptr;       // owners with copies: home dense slot
    int32_t* d_fstart = nullptr;     // n_owners + 1 entry offsets
    int32_t* d_fent = nullptr;       // per copy, in reduction order: node slot | parent << 26
    int64_t n_owners = 0;
    int max_copies = 0;
    int64_t cap_xflat = 0, cap_xflat_items = 0, cap_fent = 0, cap_fown = 0, cap_fstart = 0;
    int64_t cap_frec[3] = {0, 0, 0};
    int32_t* d_flat_pool32 = nullptr;  // scratch of the flat-table build (kept across rebuilds)
    int8_t* d_flat_pool8 = nullptr;
    int64_t cap_pool32 = 0, cap_pool8 = 0;
    int4* d_frec[3] = {nullptr, nullptr, nullptr};  // owner records: A (<=3), B (<=11), C (more)
    int64_t n_rec[3] = {0, 0, 0};
    int flat_x_e = 2;                // entries per thread of the flat coordinate kernel
    int occ_flat_x = 0;              // its resident blocks per SM at 2 entries (cached)
    int ahead_x[4] = {0, 0, 0, 0};   // resident blocks of the flat kernels (cached), by
    int ahead_f[3] = {0, 0, 0};      // entries per thread / largest tree
    // staged (MPI-era) mode: one send/receive buffer element per halo slot
    float* d_stage_buf = nullptr;
    int64_t cap_stage_buf = 0, n_stage_buf = 0;
};

namespace halo {

// halo_build.cu
// The plan's per-domain tables on the device (valid while the plan is):
// n_home[D], hstart[D] (first home-compact slot: D's home atoms in the build's
// home partition, whose ids home_gid holds), base[D] (first dense slot),
// own_off[D * (P + 1) + q] (first local index of each received slice; q = P:
// the domain's local count).
struct DomainTables {
    const int64_t* n_home;
    const int64_t* hstart;
    const int64_t* base;
    const int64_t* own_off;
};
DomainTables domain_tables(const halo_plan* pl);
int build_plan(halo_plan* pl, const float* coords, const int32_t* dom, int64_t n_atoms,
               cudaStream_t st);

int device_exclusive_scan(const int32_t* in, int32_t* out, int64_t n, int32_t* tmp,
                          cudaStream_t st);  // scratch tmp: ceil(n / kScanTile) ints

// halo_modes.cu: one launch per pulse, and the flattened exchange
int prepare_flat(halo_plan* pl, cudaStream_t st);
// The FLAT forwarding chains alone (device descriptors and sizes known); prepare_flat
// launches them itself unless this ran first in the same build.
int launch_flat_chains(halo_plan* pl, cudaStream_t st);
void free_flat(halo_plan* pl);
int launch_stepwise_x(halo_plan* pl, float* xyz, cudaStream_t st);
int launch_stepwise_f(halo_plan* pl, float* f, cudaStream_t st);
int prepare_staged(halo_plan* pl);
int launch_staged_x(halo_plan* pl, float* xyz, cudaStream_t st);
int launch_staged_f(halo_plan* pl, float* f, cudaStream_t st);
int launch_flat_x(halo_plan* pl, float* xyz, cudaStream_t st);
int launch_flat_f(halo_plan* pl, float* f, cudaStream_t st);

// halo_exchange.cu
// per-(s, p) descriptors and the error word, for every mode
int prepare_common(halo_plan* pl, cudaStream_t st);
// the FUSED mode's work lists, counters and tickets (synchronises `st`)
int prepare_fused(halo_plan* pl, cudaStream_t st);
int launch_exchange_x(halo_plan* pl, float* xyz, cudaStream_t st);
int launch_exchange_f(halo_plan* pl, float* f, cudaStream_t st);
// the coordinate kernel with caller-supplied arrival counters and ticket
// (zeroed by the caller before the launch)
int launch_exchange_x_scratch(halo_plan* pl, float* xyz, uint32_t* arrived,
                              unsigned long long* ticket, cudaStream_t st);
// the sharded data plane: the FUSED kernels with per-shard buffers and
// system-scope signals (every shard's work in one launch on this GPU)
int launch_exchange_x_sharded(halo_plan* pl, float* const* shard_xyz, cudaStream_t st);
int launch_exchange_f_sharded(halo_plan* pl, float* const* shard_f, cudaStream_t st);
int launch_load_home_sharded(const halo_plan* pl, const float* g, float* const* shard_local,
                             cudaStream_t st);
int launch_store_home_sharded(const halo_plan* pl, const float* const* shard_local, float* g,
                              cudaStream_t st);
// shard_dom from the grid (z-slabs), shard_first from the plan's layout
int set_shards(halo_plan* pl, int n_shards);
void update_shard_first(halo_plan* pl);
int launch_load_home(const halo_plan* pl, const float* g, float* local, cudaStream_t st);
int launch_store_home(const halo_plan* pl, const float* local, float* g, cudaStream_t st);
int launch_local_to_global(const halo_plan* pl, int32_t* out, cudaStream_t st);
void free_exchange(halo_plan* pl);
int reset_flags(halo_plan* pl, cudaStream_t st);

void free_build(halo_plan* pl);

// halo_noalloc.cu: stores the device address of halo_exchange_x_noalloc's
// fixed array for the current device (once per device; called by setup)
int noalloc_prepare();

inline int cuda_code(cudaError_t e) { return e == cudaSuccess ? HALO_OK : HALO_ECUDA; }

// Launch with programmatic stream serialization: the kernel may be scheduled
// while its predecessor in the stream drains, and holds back every access to
// data an earlier kernel wrote until grid_dependency_wait() (the exchange
// kernels of the flat and stepwise modes, and every kernel of the build,
// each of which starts with grid_launch_dependents() and
// grid_dependency_wait(), so the next kernel's launch overlaps the end of the
// one before).  smem: dynamic shared memory bytes.
template <class... KArgs, class... Args>
inline cudaError_t launch_dependent_shm(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                        cudaStream_t st, Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

template <class... KArgs, class... Args>
inline cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t st,
                                    Args... args) {
    return launch_dependent_shm(kernel, grid, block, 0, st, args...);
}

template <class T>
inline int dev_alloc(T** p, size_t count) {
    *p = nullptr;
    if (count == 0) count = 1;
    cudaError_t e = cudaMalloc((void**)p, count * sizeof(T));
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        *p = nullptr;
        return e == cudaErrorMemoryAllocation ? HALO_ENOMEM : HALO_ECUDA;
    }
    return HALO_OK;
}

template <class T>
inline void dev_free(T*& p) {
    if (p) cudaFree((void*)p);
    p = nullptr;
}

// Grow-only device buffer: reallocates (with 25 % headroom) only when `count`
// exceeds the capacity, so rebuilds of a plan do not free and re-allocate
// (cudaFree synchronises the device).
template <class T>
inline int dev_reserve(T** p, int64_t* cap, int64_t count) {
    if (*p && *cap >= count) return HALO_OK;
    dev_free(*p);
    *cap = 0;
    int64_t want = count < 1 ? 1 : count;
    want += want / 4;
    const int rc = dev_alloc(p, (size_t)want);
    if (rc == HALO_OK) *cap = want;
    return rc;
}

// Pinned host staging of at least `bytes` (grow-only; the stream must be idle
// when it grows, which holds at the points the build calls it).
inline int host_stage(halo_plan* pl, size_t bytes, void** out) {
    if (pl->h_stage_cap < bytes) {
        if (pl->h_stage) cudaFreeHost(pl->h_stage);
        pl->h_stage = nullptr;
        pl->h_stage_cap = 0;
        pl->h_stage_dev = nullptr;
        const size_t want = bytes + bytes / 4 + 4096;
        if (cudaHostAlloc(&pl->h_stage, want, cudaHostAllocMapped) != cudaSuccess) {
            (void)cudaGetLastError();
            pl->h_stage = nullptr;
            return HALO_ENOMEM;
        }
        pl->h_stage_cap = want;
        // kernels write the words the host reads back straight into it
        if (pl->stage_copies || cudaHostGetDevicePointer(&pl->h_stage_dev, pl->h_stage, 0) != cudaSuccess) {
            (void)cudaGetLastError();
            pl->h_stage_dev = nullptr;
        }
    }
    *out = pl->h_stage;
    return HALO_OK;
}

}  // namespace halo

#define HALO_TRY(x)                      \
    do {                                 \
        int _rc = (x);                   \
        if (_rc != HALO_OK) return _rc;  \
    } while (0)

#define HALO_CUDA(x)                              \
    do {                                          \
        cudaError_t _e = (x);                     \
        if (_e != cudaSuccess) return HALO_ECUDA; \
    } while (0)
