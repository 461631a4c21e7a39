// halo_exchange.cu -- the coordinate exchange and the force reduction, each one
// kernel launch for all pulses.
//
// Page "Redesigning GROMACS Halo Exchange: Improving Strong Scaling with
// GPU-initiated NVSHMEM" (review):
//   Algorithms 3/4 (FusedPackCommX, packWithDeps): every pulse is packed by one
//     launch; index-map entries below depOffset are gathered at once, entries
//     at or above it only after the pulses that delivered them have signalled;
//   Algorithm 5 (syncAndCommWithDeps): a block barrier, then one thread bumps
//     the pulse's completion counter with gpu-scope release semantics;
//   Algorithm 6 (FusedCommUnpackF): pulses from the last to the first, each
//     received halo force added to the slot its index-map entry names.
//
// On one GPU every domain lives in the same HBM, so the "remote" store of the
// pages is a store into the receiving domain's halo slice of the caller's dense
// buffer, and the per-pulse signal is a per-(domain, pulse) counter:
//   arrived[r*P + p]  chunks of pulse p delivered into domain r (coordinates),
//   done[s*P + p]     chunks of pulse p reduced into domain s (forces).
// A consumer waits (acquire, gpu scope) until the counter reaches
// epoch * chunks; the epoch is the call number, recovered from a monotonically
// increasing work ticket, so no counter is ever reset between calls.
//
// Work order.  Items are listed pulse by pulse (ascending for coordinates,
// descending for forces) and, within a pulse, the dependent chunks first: the
// forwarding chain is served first and the bulk of independent traffic
// streams behind it.  Coordinates: a chunk is independent when all its
// entries lie below depOffset.  Forces: the build classifies every entry; an
// entry is independent when no later pulse adds into its destination slot and
// its halo source slot was never forwarded.  Dependent force chunks wait for
// the later pulses that touch their destination domain or their source
// slice.  Each destination slot still receives its adds in reverse pulse
// order, so the result is bit-identical to the sequential reduction.
//
// Forward progress: blocks (coordinate items) and warps (force items) take
// work items from one atomic ticket counter in that order, and an item only
// waits on items with earlier tickets.  The earliest unfinished item is the
// current item of a running block or warp (each holds at most the item it
// works on and one prefetched, later ticket), and everything it waits on has
// an earlier ticket, so by induction every wait ends -- whatever the grid size
// and however blocks are scheduled.  Every wait is still bounded
// in time and reports HALO_ETIMEOUT through the plan's error word.
#include <string.h>

#include <algorithm>

#include "halo_device.cuh"
#include "halo_internal.cuh"

namespace halo {
namespace {

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// System scope: the sharded data plane, whose counters and buffers would sit
// on different GPUs ("Redesigning GROMACS Halo Exchange ...", section 4,
// memory ordering: the receiver's signal is a system-scope release store).
__device__ __forceinline__ uint32_t ld_acquire_sys(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

template <bool SYS>
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
    return SYS ? ld_acquire_sys(p) : ld_acquire_gpu(p);
}

__device__ __forceinline__ int ld_relaxed_gpu(const int* p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_gpu_add(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_release_sys_add(uint32_t* p, uint32_t v) {
    asm volatile("red.release.sys.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

template <bool SYS>
__device__ __forceinline__ void red_release_add(uint32_t* p, uint32_t v) {
    if (SYS)
        red_release_sys_add(p, v);
    else
        red_release_gpu_add(p, v);
}

// Dense slot g of shard k in the sharded data plane.
__device__ __forceinline__ float* shard_slot(const ShardTable& t, int k, int64_t g) {
    return t.ptr[k] + 3 * (g - t.first[k]);
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ unsigned smid() {
    unsigned r;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
    return r;
}

// Trace record of one work item: ticket time, time the waits ended, release
// time (global timer, ns) and the SM that ran it.
__device__ __forceinline__ void trace_item(unsigned long long* trace, int item, uint64_t t0,
                                           uint64_t t1) {
    unsigned long long* r = trace + 4 * (int64_t)item;
    r[0] = t0;
    r[1] = t1;
    r[2] = global_timer_ns();
    r[3] = smid();
}


// Bounded wait until *c has reached target (modulo 2^32).  On timeout the
// first waiter records where it gave up; every waiter gives up as soon as the
// plan's error word is set.
template <bool SYS>
__device__ bool wait_count(const uint32_t* c, uint32_t target, int* err, long long timeout_ns,
                           int kernel, int flag) {
    if ((int32_t)(ld_acquire<SYS>(c) - target) >= 0) return true;
    const uint64_t t0 = global_timer_ns();
    unsigned ns = 8;
    for (;;) {
        __nanosleep(ns);
        if (ns < 128) ns <<= 1;
        if ((int32_t)(ld_acquire<SYS>(c) - target) >= 0) return true;
        if (ld_relaxed_gpu(err) != 0) return false;
        if ((long long)(global_timer_ns() - t0) > timeout_ns) {
            if (atomicCAS(err, 0, HALO_ETIMEOUT) == 0) {
                err[1] = kernel;
                err[2] = flag;
            }
            return false;
        }
    }
}

struct XArgs {
    float* xyz;
    const int32_t* maps;
    const XItem* items;
    const uint32_t* target;  // chunks delivered into each (r, p)
    uint32_t* arrived;
    unsigned long long* ticket;
    int* err;
    int n_items;
    long long timeout_ns;
    int drop_flag;
    int64_t n_slots;  // local slots (checked in debug builds)
    unsigned long long* trace;  // optional: 4 words per item (see halo_set_trace)
    ShardTable sh;    // sharded data plane only
};

struct FArgs {
    float* f;
    const int2* pairs;
    const FItem* items;
    const uint32_t* target;  // chunks reduced into each (s, p)
    uint32_t* done;
    unsigned long long* ticket;
    int* err;
    int n_items;
    long long timeout_ns;
    unsigned long long* trace;
    int64_t n_slots;  // local slots (checked in debug builds)
    ShardTable sh;    // sharded data plane only
};

constexpr int kWarps = kThreads / 32;

// Work items are warp-granular: every warp takes its own tickets (lane 0
// draws, the value is broadcast), so a warp that waits for a pulse holds up
// no other warp -- the pages' NVLink path, where each warp packs its own chunk
// and its leader issues the bulk store (Algorithm 3).  A warp's ticket t
// decodes to call number t / T and item t mod T, with T = items + warps in
// the grid: every warp ends by drawing exactly one ticket past the items.
struct WarpTicket {
    int item;
    uint32_t epoch;
};

__device__ __forceinline__ WarpTicket decode_ticket(unsigned long long t, unsigned long long T) {
    const unsigned long long k = t / T;
    return WarpTicket{(int)(t - k * T), (uint32_t)(k + 1)};
}

// Coordinates: block-granular items of up to kThreads * E entries whose
// destination is one contiguous halo range; the block stages it in shared
// memory and one thread writes it with a single bulk copy.
// SHARDED: the sharded data plane (sources and destinations in per-shard
// buffers, system-scope signals); otherwise one dense buffer, gpu scope.
template <int E, bool SHARDED>
__global__ void __launch_bounds__(kThreads) pack_x_kernel(const __grid_constant__ XArgs a) {
    __shared__ __align__(128) float stage[3 * kThreads * E + 4];
    __shared__ unsigned long long s_ticket;
    __shared__ int s_go;
    // programmatic dependent launch: the launch overlaps the kernel before this
    // one in the stream; nothing (tickets included) is touched before it ends
    grid_launch_dependents();
    grid_dependency_wait();
    const unsigned long long T = (unsigned long long)a.n_items + gridDim.x;
    unsigned long long next = 0;
    if (threadIdx.x == 0) next = atomicAdd(a.ticket, 1ull);
    for (;;) {
        if (threadIdx.x == 0) {
            s_ticket = next;
            const WarpTicket tk0 = decode_ticket(next, T);
            s_go = tk0.item < a.n_items && ld_relaxed_gpu(a.err) == 0;
            if (s_go) next = atomicAdd(a.ticket, 1ull);  // prefetch the next ticket
        }
        __syncthreads();
        if (!s_go) return;
        const WarpTicket tk = decode_ticket(s_ticket, T);
        const uint64_t t_take = a.trace && threadIdx.x == 0 ? global_timer_ns() : 0;
        const XItem w = a.items[tk.item];
        const bool dependent = w.wait_mask != 0;
        const int32_t* map = a.maps + w.map_off;
        const float* src = SHARDED ? shard_slot(a.sh, w.src_shard, w.src_base) : a.xyz + 3 * w.src_base;
        float* dst = SHARDED ? shard_slot(a.sh, w.dst_shard, w.dst) : a.xyz + 3 * w.dst;
        // index loads first: only the forwarded coordinates remain after a wait
        int idx[E];
        const bool dst_ok = w.len <= 0 || in_range(w.dst + w.len - 1, a.n_slots, a.err);
#pragma unroll
        for (int e = 0; e < E; e++) {
            const int i = threadIdx.x + e * kThreads;
            idx[e] = i < w.len ? __ldg(map + i) : -1;
            if (idx[e] >= 0 && !(dst_ok && in_range(w.src_base + idx[e], a.n_slots, a.err)))
                idx[e] = -1;
        }
        if (dependent) {
            // packWithDeps: one thread waits for the pulses that delivered the
            // slots this chunk forwards (Algorithm 4), then the block goes on
            __syncthreads();  // every thread has read s_go / s_ticket
            if (threadIdx.x == 0) {
                int ok = 1;
                for (uint64_t m = w.wait_mask; m && ok; m &= m - 1) {
                    const int c = w.wait_base + __ffsll((long long)m) - 1;
                    ok = wait_count<SHARDED>(a.arrived + c, tk.epoch * __ldg(a.target + c), a.err,
                                             a.timeout_ns, 1, c);
                }
                s_go = ok;
            }
            __syncthreads();
            if (!s_go) return;
        }
        const uint64_t t_wait = a.trace && threadIdx.x == 0 ? global_timer_ns() : 0;
        float v[E][3];
#pragma unroll
        for (int e = 0; e < E; e++) {
            if (idx[e] >= 0) {
                const float* p = src + 3 * (int64_t)idx[e];
                if (dependent) {  // slots written by this launch: read through L2
                    v[e][0] = __ldcg(p);
                    v[e][1] = __ldcg(p + 1);
                    v[e][2] = __ldcg(p + 2);
                } else {          // home slots: read-only for the launch
                    v[e][0] = __ldg(p);
                    v[e][1] = __ldg(p + 1);
                    v[e][2] = __ldg(p + 2);
                }
            }
        }
        // stage the chunk's contiguous destination range; one thread writes
        // it with a bulk asynchronous copy (the pages' TMA store of a packed
        // chunk, Algorithm 3), then signals with a gpu-scope release
        // (Algorithm 5)
        const int sh = stage_shift(dst);
#pragma unroll
        for (int e = 0; e < E; e++) {
            if (idx[e] >= 0) {
                float* q = stage + sh + 3 * (threadIdx.x + e * kThreads);
                q[0] = v[e][0] + w.shift[0];
                q[1] = v[e][1] + w.shift[1];
                q[2] = v[e][2] + w.shift[2];
            }
        }
        fence_smem_to_async();
        __syncthreads();
        if (threadIdx.x == 0) {
            if (dst_ok) bulk_store_floats(dst, stage, 3 * w.len, true);
            if (w.flag != a.drop_flag) red_release_add<SHARDED>(a.arrived + w.flag, 1u);
            if (a.trace) trace_item(a.trace, tk.item, t_take, t_wait);
        }
        // the next iteration's barrier keeps the stage until the copy has read it
    }
}

template <int E, bool SHARDED>
__global__ void __launch_bounds__(kThreads, 4) unpack_f_kernel(const __grid_constant__ FArgs a) {
    const int lane = threadIdx.x & 31;
    grid_launch_dependents();  // as in pack_x_kernel
    grid_dependency_wait();
    const unsigned long long T = (unsigned long long)a.n_items + (unsigned long long)gridDim.x * kWarps;
    unsigned long long next = 0;
    if (lane == 0) next = atomicAdd(a.ticket, 1ull);
    next = __shfl_sync(kFull, next, 0);
    for (;;) {
        const WarpTicket tk = decode_ticket(next, T);
        if (tk.item >= a.n_items) return;
        int stop = 0;
        if (lane == 0) {
            stop = ld_relaxed_gpu(a.err) != 0;
            if (!stop) next = atomicAdd(a.ticket, 1ull);
        }
        if (__shfl_sync(kFull, stop, 0)) return;
        const uint64_t t_take = a.trace && lane == 0 ? global_timer_ns() : 0;
        const FItem w = a.items[tk.item];
        const int2* pr = a.pairs + w.off;
        int2 sd[E];
#pragma unroll
        for (int e = 0; e < E; e++) {
            const int i = lane + 32 * e;
            sd[e] = i < w.len ? __ldg(pr + i) : make_int2(-1, -1);
            if (sd[e].x >= 0 && !(in_range(sd[e].x, a.n_slots, a.err) &&
                                  in_range(sd[e].y, a.n_slots, a.err)))
                sd[e] = make_int2(-1, -1);
        }
        // halo sources in r's shard, destinations in s's shard (one buffer
        // when not sharded)
        const float* fr = SHARDED ? a.sh.ptr[w.r_shard] : a.f;
        float* fs = SHARDED ? a.sh.ptr[w.s_shard] : a.f;
        const int64_t r0 = SHARDED ? a.sh.first[w.r_shard] : 0;
        const int64_t s0 = SHARDED ? a.sh.first[w.s_shard] : 0;
        if (w.ms | w.mr) {
            // warm L2 with the lines read after the wait (L2 is coherent, so
            // the loads that follow the acquire still see the latest values);
            // sharded: only the destination lines, which are s's own
#pragma unroll
            for (int e = 0; e < E; e++) {
                if (sd[e].x >= 0) {
                    if (!SHARDED) prefetch_l2(fr + 3 * ((int64_t)sd[e].x - r0));
                    prefetch_l2(fs + 3 * ((int64_t)sd[e].y - s0));
                }
            }
            int ok = 1;
            if (lane == 0) {
                for (uint64_t m = w.ms; m && ok; m &= m - 1) {
                    const int c = w.s_base + __ffsll((long long)m) - 1;
                    ok = wait_count<SHARDED>(a.done + c, tk.epoch * __ldg(a.target + c), a.err,
                                             a.timeout_ns, 2, c);
                }
                for (uint64_t m = w.mr; m && ok; m &= m - 1) {
                    const int c = w.r_base + __ffsll((long long)m) - 1;
                    ok = wait_count<SHARDED>(a.done + c, tk.epoch * __ldg(a.target + c), a.err,
                                             a.timeout_ns, 2, c);
                }
            }
            if (!__shfl_sync(kFull, ok, 0)) return;
        }
        const uint64_t t_wait = a.trace && lane == 0 ? global_timer_ns() : 0;
        float h[E][3], o[E][3];
#pragma unroll
        for (int e = 0; e < E; e++) {
            if (sd[e].x >= 0) {
                const float* hp = fr + 3 * ((int64_t)sd[e].x - r0);
                const float* op = fs + 3 * ((int64_t)sd[e].y - s0);
                h[e][0] = __ldcg(hp);
                h[e][1] = __ldcg(hp + 1);
                h[e][2] = __ldcg(hp + 2);
                o[e][0] = __ldcg(op);
                o[e][1] = __ldcg(op + 1);
                o[e][2] = __ldcg(op + 2);
            }
        }
#pragma unroll
        for (int e = 0; e < E; e++) {
            if (sd[e].x >= 0) {
                float* op = fs + 3 * ((int64_t)sd[e].y - s0);
                op[0] = o[e][0] + h[e][0];
                op[1] = o[e][1] + h[e][1];
                op[2] = o[e][2] + h[e][2];
            }
        }
        // the warp's stores, then one release by the leader (gpu scope; system
        // scope on the sharded data plane)
        __syncwarp();
        if (lane == 0) {
            red_release_add<SHARDED>(a.done + w.flag, 1u);
            if (a.trace) trace_item(a.trace, tk.item, t_take, t_wait);
        }
        next = __shfl_sync(kFull, next, 0);
    }
}

// ---- build-time kernels of the exchange plan --------------------------------------

// wmax[dense slot] = last pulse whose index map names the slot (pulses are
// launched in ascending order; within one pulse a slot appears at most once).
__global__ void mark_kernel(const SPDesc* __restrict__ sp, const int32_t* __restrict__ maps,
                            int8_t* __restrict__ wmax, int P, int p) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    const SPDesc d = sp[(int64_t)blockIdx.y * P + p];
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < d.send; i += gridDim.x * blockDim.x)
        wmax[d.src_base + maps[d.map_off + i]] = (int8_t)p;
}

// Stable partition of the force entries of one (s, p) into independent then
// dependent, written as (source halo slot, destination slot) pairs.
__global__ void __launch_bounds__(kThreads) classify_kernel(const SPDesc* __restrict__ sp,
                                                            const int32_t* __restrict__ maps,
                                                            const int8_t* __restrict__ wmax,
                                                            int2* __restrict__ pairs,
                                                            int32_t* __restrict__ nindep) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    __shared__ int wi[kThreads / 32], wd[kThreads / 32];
    __shared__ int s_tot;
    const SPDesc d = sp[blockIdx.x];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned lt = lanemask_lt();
    int cnt = 0;
    for (int i = threadIdx.x; i < d.send; i += kThreads) {
        const int64_t dst = d.src_base + maps[d.map_off + i];
        const int64_t src = d.dst + i;
        cnt += (wmax[dst] == d.p && wmax[src] < 0) ? 1 : 0;
    }
    cnt = __reduce_add_sync(kFull, cnt);
    if (lane == 0) wi[warp] = cnt;
    __syncthreads();
    if (threadIdx.x == 0) {
        int t = 0;
        for (int w = 0; w < kThreads / 32; w++) t += wi[w];
        s_tot = t;
        nindep[blockIdx.x] = t;
    }
    __syncthreads();
    int oi = 0, od = s_tot;
    for (int b = 0; b < d.send; b += kThreads) {
        const int i = b + threadIdx.x;
        bool ind = false;
        int2 v = make_int2(0, 0);
        const bool valid = i < d.send;
        if (valid) {
            const int64_t dst = d.src_base + maps[d.map_off + i];
            const int64_t src = d.dst + i;
            ind = wmax[dst] == d.p && wmax[src] < 0;
            v = make_int2((int)src, (int)dst);
        }
        const unsigned bi = __ballot_sync(kFull, valid && ind);
        const unsigned bd = __ballot_sync(kFull, valid && !ind);
        __syncthreads();
        if (lane == 0) {
            wi[warp] = __popc(bi);
            wd[warp] = __popc(bd);
        }
        __syncthreads();
        int pi = 0, pd = 0, ti = 0, td = 0;
#pragma unroll
        for (int w = 0; w < kThreads / 32; w++) {
            pi += w < warp ? wi[w] : 0;
            pd += w < warp ? wd[w] : 0;
            ti += wi[w];
            td += wd[w];
        }
        if (valid) {
            const int pos = ind ? oi + pi + __popc(bi & lt) : od + pd + __popc(bd & lt);
            pairs[d.map_off + pos] = v;
        }
        oi += ti;
        od += td;
    }
}

// Home atoms: block (x, D) takes domain D's home atoms j = x * blockDim +
// thread, striding by gridDim.x * blockDim; atom home_gid[hstart[D] + j]
// (the home partition) sits at dense slot base[D] + j.
__global__ void load_home_kernel(DomainTables t, const int32_t* __restrict__ home_gid, int64_t n,
                                 const float* __restrict__ g, float* __restrict__ local,
                                 int64_t n_slots, int* err) {
    const int D = blockIdx.y;
    const int64_t h0 = t.hstart[D], nh = t.n_home[D], b = t.base[D];
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < nh;
         j += (int64_t)gridDim.x * blockDim.x) {
        const int64_t dd = b + j, a = home_gid[h0 + j];
        if (!in_range(dd, n_slots, err) || !in_range(a, n, err)) continue;
        local[3 * dd + 0] = g[3 * a + 0];
        local[3 * dd + 1] = g[3 * a + 1];
        local[3 * dd + 2] = g[3 * a + 2];
    }
}

__global__ void store_home_kernel(DomainTables t, const int32_t* __restrict__ home_gid, int64_t n,
                                  const float* __restrict__ local, float* __restrict__ g,
                                  int64_t n_slots, int* err) {
    const int D = blockIdx.y;
    const int64_t h0 = t.hstart[D], nh = t.n_home[D], b = t.base[D];
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < nh;
         j += (int64_t)gridDim.x * blockDim.x) {
        const int64_t dd = b + j, a = home_gid[h0 + j];
        if (!in_range(dd, n_slots, err) || !in_range(a, n, err)) continue;
        g[3 * a + 0] = local[3 * dd + 0];
        g[3 * a + 1] = local[3 * dd + 1];
        g[3 * a + 2] = local[3 * dd + 2];
    }
}

// Sharded data plane: the shard holding dense slot dd (shards are contiguous
// ranges of dense slots, so a domain lies in one).
__device__ __forceinline__ int shard_of_slot(const ShardTable& t, int n_shards, int64_t dd) {
    int k = 0;
    while (k + 1 < n_shards && dd >= t.first[k + 1]) k++;
    return k;
}

__global__ void load_home_sharded_kernel(DomainTables t, const int32_t* __restrict__ home_gid,
                                         int64_t n, const float* __restrict__ g,
                                         const __grid_constant__ ShardTable sh, int n_shards,
                                         int64_t n_slots, int* err) {
    const int D = blockIdx.y;
    const int64_t h0 = t.hstart[D], nh = t.n_home[D], b = t.base[D];
    const int k = shard_of_slot(sh, n_shards, b);
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < nh;
         j += (int64_t)gridDim.x * blockDim.x) {
        const int64_t dd = b + j, a = home_gid[h0 + j];
        if (!in_range(dd, n_slots, err) || !in_range(a, n, err)) continue;
        float* q = sh.ptr[k] + 3 * (dd - sh.first[k]);
        q[0] = g[3 * a + 0];
        q[1] = g[3 * a + 1];
        q[2] = g[3 * a + 2];
    }
}

__global__ void store_home_sharded_kernel(DomainTables t, const int32_t* __restrict__ home_gid,
                                          int64_t n, const __grid_constant__ ShardTable sh,
                                          int n_shards, float* __restrict__ g, int64_t n_slots,
                                          int* err) {
    const int D = blockIdx.y;
    const int64_t h0 = t.hstart[D], nh = t.n_home[D], b = t.base[D];
    const int k = shard_of_slot(sh, n_shards, b);
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < nh;
         j += (int64_t)gridDim.x * blockDim.x) {
        const int64_t dd = b + j, a = home_gid[h0 + j];
        if (!in_range(dd, n_slots, err) || !in_range(a, n, err)) continue;
        const float* q = sh.ptr[k] + 3 * (dd - sh.first[k]);
        g[3 * a + 0] = q[0];
        g[3 * a + 1] = q[1];
        g[3 * a + 2] = q[2];
    }
}

__global__ void home_gid_kernel(DomainTables t, const int32_t* __restrict__ home_gid,
                                int32_t* __restrict__ out) {
    const int D = blockIdx.y;
    const int64_t h0 = t.hstart[D], nh = t.n_home[D], b = t.base[D];
    for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < nh;
         j += (int64_t)gridDim.x * blockDim.x)
        out[b + j] = home_gid[h0 + j];
}

// Owner id of every halo slot of one pulse.
__global__ void halo_gid_kernel(const SPDesc* __restrict__ sp, const int32_t* __restrict__ maps,
                                int32_t* out, int P, int p) {
    const SPDesc d = sp[(int64_t)blockIdx.y * P + p];
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < d.send; i += gridDim.x * blockDim.x)
        out[d.dst + i] = out[d.src_base + maps[d.map_off + i]];
}

// ---- work lists, generated on the device ------------------------------------
// Groups of chunks, in ticket order.  Coordinates: for p ascending, the
// dependent chunks of every sender, then the independent ones.  Forces: for p
// descending, the dependent chunks of every sender, then the independent ones.
struct ItemGen {
    const SPDesc* sp;
    const int32_t* nindep;          // independent force entries per (s, p)
    const uint64_t* recv_mask;      // per domain: pulses that delivered a nonempty slice
    int nd, P, CH, CHF;
    int n_shards;
    int shard_dom[kMaxShards + 1];  // shard k holds domains [shard_dom[k], shard_dom[k + 1])
    uint64_t fms[HALO_MAX_PULSES];  // force waits on s per pulse
    uint64_t fmr[HALO_MAX_PULSES];  // force waits on r per pulse
};

__global__ void recv_mask_kernel(const SPDesc* __restrict__ sp, int nsp, uint64_t* mask) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nsp; i += gridDim.x * blockDim.x) {
        const SPDesc d = sp[i];
        if (d.send > 0) atomicOr((unsigned long long*)(mask + d.r), 1ull << d.p);
    }
}

__device__ __forceinline__ int16_t shard_of(const ItemGen& a, int D) {
    int k = 0;
    while (k + 1 < a.n_shards && D >= a.shard_dom[k + 1]) k++;
    return (int16_t)k;
}

// Group g of the coordinate list: p = g / (2 nd), dependent first, sender s.
__device__ __forceinline__ void x_group(const ItemGen& a, int g, int* sp, int* lo, int* hi, bool* dep) {
    const int p = g / (2 * a.nd), s = g % a.nd;
    *dep = ((g / a.nd) % 2) == 0;
    *sp = s * a.P + p;
    const SPDesc& d = a.sp[*sp];
    *lo = *dep ? d.split : 0;
    *hi = *dep ? d.send : d.split;
}

// Group g of the force list: p = P - 1 - g / (2 nd), dependent first, sender s.
__device__ __forceinline__ void f_group(const ItemGen& a, int g, int* sp, int* lo, int* hi, bool* dep) {
    const int p = a.P - 1 - g / (2 * a.nd), s = g % a.nd;
    *dep = ((g / a.nd) % 2) == 0;
    *sp = s * a.P + p;
    const int ni = a.nindep[*sp];
    *lo = *dep ? ni : 0;
    *hi = *dep ? a.sp[*sp].send : ni;
}

__global__ void item_count_kernel(ItemGen a, int32_t* cx, int32_t* cf, uint32_t* target) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    const int ng = 2 * a.P * a.nd;
    for (int g = blockIdx.x * blockDim.x + threadIdx.x; g < ng; g += gridDim.x * blockDim.x) {
        int sp, lo, hi;
        bool dep;
        x_group(a, g, &sp, &lo, &hi, &dep);
        cx[g] = (hi - lo + a.CH - 1) / a.CH;
        f_group(a, g, &sp, &lo, &hi, &dep);
        cf[g] = (hi - lo + a.CHF - 1) / a.CHF;
    }
    const int nsp = a.P * a.nd;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nsp; i += gridDim.x * blockDim.x) {
        const SPDesc d = a.sp[i];
        const int ni = a.nindep[i];
        target[d.r * a.P + d.p] = (uint32_t)((d.split + a.CH - 1) / a.CH +
                                             (d.send - d.split + a.CH - 1) / a.CH);
        target[nsp + i] = (uint32_t)((ni + a.CHF - 1) / a.CHF + (d.send - ni + a.CHF - 1) / a.CHF);
    }
}

__global__ void item_fill_kernel(ItemGen a, const int32_t* __restrict__ bx,
                                 const int32_t* __restrict__ bf, XItem* __restrict__ ix,
                                 FItem* __restrict__ iff) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    const int g = blockIdx.x;
    int sp, lo, hi;
    bool dep;
    x_group(a, g, &sp, &lo, &hi, &dep);
    {
        const SPDesc d = a.sp[sp];
        const uint64_t below = d.p > 0 ? (~0ull >> (64 - d.p)) : 0ull;
        const uint64_t mask = dep ? (a.recv_mask[d.s] & below) : 0ull;
        const int n = (hi - lo + a.CH - 1) / a.CH;
        for (int c = threadIdx.x; c < n; c += blockDim.x) {
            const int st0 = lo + c * a.CH;
            XItem w;
            w.map_off = d.map_off + st0;
            w.src_base = d.src_base;
            w.dst = d.dst + st0;
            w.len = min(a.CH, hi - st0);
            w.flag = d.r * a.P + d.p;
            w.wait_base = d.s * a.P;
            w.src_shard = shard_of(a, d.s);
            w.dst_shard = shard_of(a, d.r);
            w.wait_mask = mask;
            w.shift[0] = d.shift[0];
            w.shift[1] = d.shift[1];
            w.shift[2] = d.shift[2];
            w.pad2 = 0;
            ix[bx[g] + c] = w;
        }
    }
    f_group(a, g, &sp, &lo, &hi, &dep);
    {
        const SPDesc d = a.sp[sp];
        const bool waits = dep && (a.fms[d.p] | a.fmr[d.p]) != 0;
        const int n = (hi - lo + a.CHF - 1) / a.CHF;
        for (int c = threadIdx.x; c < n; c += blockDim.x) {
            const int st0 = lo + c * a.CHF;
            FItem w;
            w.off = d.map_off + st0;
            w.len = min(a.CHF, hi - st0);
            w.flag = d.s * a.P + d.p;
            w.s_base = d.s * a.P;
            w.r_base = d.r * a.P;
            w.ms = waits ? a.fms[d.p] : 0ull;
            w.mr = waits ? a.fmr[d.p] : 0ull;
            w.s_shard = shard_of(a, d.s);
            w.r_shard = shard_of(a, d.r);
            w.pad = 0;
            iff[bf[g] + c] = w;
        }
    }
}

int grid_cells(const halo_plan* pl, int D, int c[3]) {
    c[0] = D % pl->grid[0];
    c[1] = (D / pl->grid[0]) % pl->grid[1];
    c[2] = D / (pl->grid[0] * pl->grid[1]);
    return 0;
}

template <int E>
int occupancy(int* blocks_x, int* blocks_f) {
    // the sharded variants have the same resources (checked by the build's register report)
    HALO_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_x, pack_x_kernel<E, false>, kThreads, 0));
    HALO_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_f, unpack_f_kernel<E, false>, kThreads, 0));
    return HALO_OK;
}

}  // namespace

void free_exchange(halo_plan* pl) {
    dev_free(pl->d_sp);
    dev_free(pl->d_items_x);
    dev_free(pl->d_items_f);
    dev_free(pl->d_fpairs);
    dev_free(pl->d_wmax);
    dev_free(pl->d_nindep);
    dev_free(pl->d_target);
    dev_free(pl->d_flags);
    dev_free(pl->d_tickets);
    dev_free(pl->d_err);
    dev_free(pl->d_recv_mask);
    dev_free(pl->d_itemgen);
    pl->cap_recv_mask = pl->cap_itemgen = 0;
    pl->fpairs_cap = 0;
    pl->wmax_cap = 0;
    pl->cap_sp = pl->cap_items_x = pl->cap_items_f = pl->cap_target = pl->cap_flags = 0;
    pl->cap_nindep = 0;
}

int reset_flags(halo_plan* pl, cudaStream_t st) {
    const int nd = pl->n_dom, P = pl->P;
    if (pl->d_flags)
        HALO_CUDA(cudaMemsetAsync(pl->d_flags, 0, sizeof(uint32_t) * 2 * (size_t)nd * std::max(P, 1), st));
    if (pl->d_tickets) HALO_CUDA(cudaMemsetAsync(pl->d_tickets, 0, sizeof(unsigned long long) * 2, st));
    if (pl->d_err) HALO_CUDA(cudaMemsetAsync(pl->d_err, 0, sizeof(int) * 8, st));
    return HALO_OK;
}

int prepare_common(halo_plan* pl, cudaStream_t st) {
    const int nd = pl->n_dom, P = pl->P;
    pl->fused_ready = false;  // the FUSED work lists describe the previous plan
    if (pl->n_local_total >= ((int64_t)1 << 31)) return HALO_ECAPACITY;  // int32 dense slots
    // coordinate items: one block, kThreads * E entries; force items: one
    // warp, 32 * E entries
    const int E = 4;
    pl->entries_per_thread = E;
    pl->chunk = kThreads * E;

    // the home load / store kernels: blocks per domain so that the largest
    // domain's threads take about four atoms each
    int64_t max_home = 1;
    for (int D = 0; D < nd; D++) max_home = std::max<int64_t>(max_home, pl->n_home[D]);
    pl->home_grid_x = (int)std::min<int64_t>((max_home + 1023) / 1024, 65535);
    // the host's copy of the per (s, p) descriptors (the build wrote the
    // device's, and the largest chunk counts)
    pl->sp.assign((size_t)nd * P, SPDesc{});
    for (int s = 0; s < nd; s++) {
        int c[3];
        grid_cells(pl, s, c);
        for (int p = 0; p < P; p++) {
            const int d = pl->pulse_dim[p];
            int rc_[3] = {c[0], c[1], c[2]};
            rc_[d] = (c[d] - 1 + pl->grid[d]) % pl->grid[d];
            const int r = rc_[0] + pl->grid[0] * (rc_[1] + pl->grid[1] * rc_[2]);
            const size_t sp = (size_t)s * P + p;
            SPDesc& x = pl->sp[sp];
            x.map_off = pl->map_off[sp];
            x.src_base = pl->base[s];
            x.dst = pl->base[r] + pl->own_off[(size_t)r * (P + 1) + p];
            x.send = pl->send[sp];
            x.split = pl->split[sp];
            x.s = s;
            x.r = r;
            x.p = p;
            x.shift[0] = x.shift[1] = x.shift[2] = 0.0f;
            if (c[d] == 0) x.shift[d] = pl->box[d];
        }
    }
    if (!pl->d_err) HALO_TRY(dev_alloc(&pl->d_err, 8));
    HALO_CUDA(cudaMemsetAsync(pl->d_err, 0, sizeof(int) * 8, st));
    return HALO_OK;
}

namespace {
// The work-list totals for the host: items = the last group's offset plus its
// count, coordinate and force lists, into the host's mapped staging.
__global__ void item_totals_kernel(const int32_t* __restrict__ bx, const int32_t* __restrict__ cx,
                                   const int32_t* __restrict__ bf, const int32_t* __restrict__ cf, int ng,
                                   int32_t* __restrict__ out) {
    grid_launch_dependents();
    grid_dependency_wait();
    if (threadIdx.x == 0) {
        out[0] = bx[ng - 1] + cx[ng - 1];
        out[1] = bf[ng - 1] + cf[ng - 1];
    }
}
}  // namespace

int prepare_fused(halo_plan* pl, cudaStream_t st) {
    const int nd = pl->n_dom, P = pl->P;
    pl->trace = nullptr;  // item counts change: the caller re-arms tracing
    pl->trace_cap = 0;
    const size_t nsp = (size_t)nd * std::max(P, 1);
    const int E = pl->entries_per_thread;
    const int CHF = 32 * E;
    const int CH = pl->chunk;
    // the two list totals read back below, in the pinned staging (no copy
    // from it is in flight: every build step that uses it synchronises
    // before returning)
    int32_t* h_tot = nullptr;
    {
        void* hs = nullptr;
        HALO_TRY(host_stage(pl, 64, &hs));
        h_tot = static_cast<int32_t*>(hs);
    }

    // force-entry classification on the device: last pulse adding into each
    // slot, then a stable independent/dependent partition per (s, p)
    HALO_TRY(dev_reserve(&pl->d_nindep, &pl->cap_nindep, (int64_t)nsp));
    if (P > 0) {
        HALO_TRY(dev_reserve(&pl->d_wmax, &pl->wmax_cap, pl->n_local_total));
        HALO_TRY(dev_reserve(&pl->d_fpairs, &pl->fpairs_cap, pl->n_halo_total));
        HALO_CUDA(cudaMemsetAsync(pl->d_wmax, 0xff, (size_t)pl->n_local_total, st));
        for (int p = 0; p < P; p++) {
            const unsigned gx = (unsigned)std::min(std::max(pl->max_chunks[p], 1), 1024);
            HALO_CUDA(launch_dependent_shm(mark_kernel, dim3(gx, nd), dim3(kThreads), 0, st,
                                           (const SPDesc*)pl->d_sp, (const int32_t*)pl->d_maps, pl->d_wmax,
                                           P, p));
        }
        HALO_CUDA(launch_dependent_shm(classify_kernel, dim3((unsigned)(nd * P)), dim3(kThreads), 0, st,
                                       (const SPDesc*)pl->d_sp, (const int32_t*)pl->d_maps,
                                       (const int8_t*)pl->d_wmax, pl->d_fpairs, pl->d_nindep));
    }

    // work lists on the device: chunk counts per group, scans, fill
    const int ng = 2 * P * nd;
    ItemGen a;
    a.sp = pl->d_sp;
    a.nindep = pl->d_nindep;
    a.nd = nd;
    a.P = P;
    a.CH = CH;
    a.CHF = CHF;
    a.n_shards = pl->n_shards;
    for (int k = 0; k <= kMaxShards; k++) a.shard_dom[k] = pl->shard_dom[k];
    for (int p = 0; p < HALO_MAX_PULSES; p++) a.fms[p] = a.fmr[p] = 0;
    // dependent force entries of (s, p) wait for (s, q) and (r, q), q > p,
    // whose index maps can touch the same slots: pulse 0 of a later dim (its
    // candidates include every earlier slot) and, on r, the next pulse of the
    // same dim (its candidates are exactly this pulse's slice)
    for (int p = 0; p < P; p++)
        for (int q = p + 1; q < P; q++) {
            if (pl->pulse_k[q] == 0) {
                a.fms[p] |= 1ull << q;
                a.fmr[p] |= 1ull << q;
            } else if (q == p + 1) {
                a.fmr[p] |= 1ull << q;
            }
        }
    HALO_TRY(dev_reserve(&pl->d_target, &pl->cap_target, (int64_t)(2 * nsp)));
    HALO_TRY(dev_reserve(&pl->d_recv_mask, &pl->cap_recv_mask, (int64_t)nd));
    const int64_t nsc = (int64_t)ng / kScanTile + 2;
    HALO_TRY(dev_reserve(&pl->d_itemgen, &pl->cap_itemgen, 4 * (int64_t)std::max(ng, 1) + nsc));
    int32_t* cx = pl->d_itemgen;
    int32_t* cf = cx + std::max(ng, 1);
    int32_t* bx = cf + std::max(ng, 1);
    int32_t* bf = bx + std::max(ng, 1);
    int32_t* sct = bf + std::max(ng, 1);
    const int64_t ub_x = pl->n_halo_total / CH + ng + 1, ub_f = pl->n_halo_total / CHF + ng + 1;
    HALO_TRY(dev_reserve(&pl->d_items_x, &pl->cap_items_x, ub_x));
    HALO_TRY(dev_reserve(&pl->d_items_f, &pl->cap_items_f, ub_f));
    a.recv_mask = pl->d_recv_mask;
    // the exchanges' signal counters and tickets, cleared before the one
    // synchronisation
    HALO_TRY(dev_reserve(&pl->d_flags, &pl->cap_flags, (int64_t)(2 * nsp)));
    if (!pl->d_tickets) HALO_TRY(dev_alloc(&pl->d_tickets, 2));
    h_tot[0] = h_tot[1] = 0;
    if (ng > 0) {
        HALO_CUDA(cudaMemsetAsync(pl->d_recv_mask, 0, sizeof(uint64_t) * nd, st));
        HALO_CUDA(launch_dependent_shm(recv_mask_kernel, dim3((unsigned)((nsp + 255) / 256)), dim3(256), 0, st,
                                       (const SPDesc*)pl->d_sp, (int)nsp, pl->d_recv_mask));
        HALO_CUDA(launch_dependent_shm(item_count_kernel, dim3((unsigned)((ng + 255) / 256)), dim3(256), 0,
                                       st, a, cx, cf, pl->d_target));
        HALO_TRY(device_exclusive_scan(cx, bx, ng, sct, st));
        HALO_TRY(device_exclusive_scan(cf, bf, ng, sct, st));
        HALO_CUDA(launch_dependent_shm(item_fill_kernel, dim3((unsigned)ng), dim3(128), 0, st, a,
                                       (const int32_t*)bx, (const int32_t*)bf, pl->d_items_x,
                                       pl->d_items_f));
        // the totals come back through the mapped staging, else with copies
        if (pl->h_stage_dev) {
            HALO_CUDA(launch_dependent_shm(item_totals_kernel, dim3(1), dim3(32), 0, st, (const int32_t*)bx,
                                           (const int32_t*)cx, (const int32_t*)bf, (const int32_t*)cf, ng,
                                           static_cast<int32_t*>(pl->h_stage_dev)));
        } else {
            HALO_CUDA(cudaMemcpyAsync(h_tot + 2, bx + ng - 1, 4, cudaMemcpyDeviceToHost, st));
            HALO_CUDA(cudaMemcpyAsync(h_tot + 3, cx + ng - 1, 4, cudaMemcpyDeviceToHost, st));
            HALO_CUDA(cudaMemcpyAsync(h_tot + 4, bf + ng - 1, 4, cudaMemcpyDeviceToHost, st));
            HALO_CUDA(cudaMemcpyAsync(h_tot + 5, cf + ng - 1, 4, cudaMemcpyDeviceToHost, st));
        }
    }
    HALO_TRY(reset_flags(pl, st));
    HALO_CUDA(cudaStreamSynchronize(st));
    if (ng > 0 && !pl->h_stage_dev) {
        h_tot[0] = h_tot[2] + h_tot[3];
        h_tot[1] = h_tot[4] + h_tot[5];
    }
    pl->n_items_x = h_tot[0];
    pl->n_items_f = h_tot[1];
    if (pl->occ_x <= 0 || pl->occ_f <= 0) HALO_TRY(occupancy<4>(&pl->occ_x, &pl->occ_f));
    pl->grid_x = (int)std::max<int64_t>(
        1, std::min<int64_t>(pl->n_items_x, (int64_t)pl->num_sms * std::max(pl->occ_x, 1)));
    pl->grid_f = (int)std::max<int64_t>(
        1, std::min<int64_t>((pl->n_items_f + kWarps - 1) / kWarps,
                             (int64_t)pl->num_sms * std::max(pl->occ_f, 1)));
    pl->fused_ready = true;
    return HALO_OK;
}

int launch_exchange_x(halo_plan* pl, float* xyz, cudaStream_t st) {
    if (!pl->fused_ready) return HALO_EINVAL;
    if (pl->n_items_x == 0) return HALO_OK;
    XArgs a;
    a.xyz = xyz;
    a.maps = pl->d_maps;
    a.items = pl->d_items_x;
    a.target = pl->d_target;
    a.arrived = pl->d_flags;
    a.ticket = pl->d_tickets;
    a.err = pl->d_err;
    a.n_items = pl->n_items_x;
    a.timeout_ns = pl->wait_timeout_ns;
    a.n_slots = pl->n_local_total;
    a.drop_flag = pl->drop_flag;
    a.trace = pl->trace;
    pl->drop_flag = -1;
    const cudaError_t e = launch_dependent(pack_x_kernel<4, false>, dim3(pl->grid_x), dim3(kThreads), st, a);
    if (e != cudaSuccess) return cuda_code(e);
    pl->launches_x++;
    return HALO_OK;
}

int launch_exchange_x_scratch(halo_plan* pl, float* xyz, uint32_t* arrived,
                              unsigned long long* ticket, cudaStream_t st) {
    if (!pl->fused_ready) return HALO_EINVAL;
    if (pl->n_items_x == 0) return HALO_OK;
    XArgs a;
    a.xyz = xyz;
    a.maps = pl->d_maps;
    a.items = pl->d_items_x;
    a.target = pl->d_target;
    a.arrived = arrived;
    a.ticket = ticket;
    a.err = pl->d_err;
    a.n_items = pl->n_items_x;
    a.timeout_ns = pl->wait_timeout_ns;
    a.n_slots = pl->n_local_total;
    a.drop_flag = pl->drop_flag;
    a.trace = pl->trace;
    pl->drop_flag = -1;
    const cudaError_t e = launch_dependent(pack_x_kernel<4, false>, dim3(pl->grid_x), dim3(kThreads), st, a);
    if (e != cudaSuccess) return cuda_code(e);
    pl->launches_x++;
    return HALO_OK;
}

int launch_exchange_f(halo_plan* pl, float* f, cudaStream_t st) {
    if (!pl->fused_ready) return HALO_EINVAL;
    if (pl->n_items_f == 0) return HALO_OK;
    const size_t nsp = (size_t)pl->n_dom * std::max(pl->P, 1);
    FArgs a;
    a.f = f;
    a.pairs = pl->d_fpairs;
    a.items = pl->d_items_f;
    a.target = pl->d_target + nsp;
    a.done = pl->d_flags + nsp;
    a.ticket = pl->d_tickets + 1;
    a.err = pl->d_err;
    a.n_items = pl->n_items_f;
    a.timeout_ns = pl->wait_timeout_ns;
    a.n_slots = pl->n_local_total;
    a.trace = pl->trace ? pl->trace + 4 * (size_t)pl->n_items_x : nullptr;
    const cudaError_t e = launch_dependent(unpack_f_kernel<4, false>, dim3(pl->grid_f), dim3(kThreads), st, a);
    if (e != cudaSuccess) return cuda_code(e);
    pl->launches_f++;
    return HALO_OK;
}

int launch_store_home(const halo_plan* pl, const float* local, float* g, cudaStream_t st) {
    store_home_kernel<<<dim3(pl->home_grid_x, pl->n_dom), 256, 0, st>>>(
        domain_tables(pl), pl->d_home_gid, pl->n_atoms, local, g, pl->n_local_total, pl->d_err);
    return cuda_code(cudaGetLastError());
}

int launch_load_home(const halo_plan* pl, const float* g, float* local, cudaStream_t st) {
    load_home_kernel<<<dim3(pl->home_grid_x, pl->n_dom), 256, 0, st>>>(
        domain_tables(pl), pl->d_home_gid, pl->n_atoms, g, local, pl->n_local_total, pl->d_err);
    return cuda_code(cudaGetLastError());
}

int launch_local_to_global(const halo_plan* pl, int32_t* out, cudaStream_t st) {
    home_gid_kernel<<<dim3(pl->home_grid_x, pl->n_dom), 256, 0, st>>>(domain_tables(pl), pl->d_home_gid,
                                                                       out);
    for (int p = 0; p < pl->P; p++) {
        const unsigned gx = (unsigned)std::min(std::max(pl->max_chunks[p], 1), 1024);
        halo_gid_kernel<<<dim3(gx, pl->n_dom), kThreads, 0, st>>>(pl->d_sp, pl->d_maps, out,
                                                                   pl->P, p);
    }
    return cuda_code(cudaGetLastError());
}

// ---- sharded data plane ------------------------------------------------------------
// The pages put the domains of one system on several GPUs: a pulse whose
// receiver sits on another GPU stores the packed coordinates into that GPU's
// halo slice and signals it with a system-scope release ("Redesigning GROMACS
// Halo Exchange ...", section 3, NVLink path; section 4, memory ordering), and
// the force pass reads the remote halo forces back.  Here the plan's domains
// are split into z-slabs (shards), each with its own buffer, and the FUSED
// work lists carry every item's source and destination shard.  On one GPU
// every shard's items run in one launch, in ticket order, so the waits between
// shards resolve by the same induction as in the FUSED mode.

int set_shards(halo_plan* pl, int n_shards) {
    const int nz = pl->grid[2];
    if (n_shards < 1 || n_shards > kMaxShards || n_shards > nz) return HALO_EINVAL;
    const int layer = pl->grid[0] * pl->grid[1];
    pl->n_shards = n_shards;
    for (int k = 0; k <= kMaxShards; k++) {
        const int kk = std::min(k, n_shards);
        pl->shard_dom[k] = (int)(((int64_t)kk * nz / n_shards) * layer);
    }
    update_shard_first(pl);
    return HALO_OK;
}

void update_shard_first(halo_plan* pl) {
    for (int k = 0; k <= kMaxShards; k++) {
        const int D = pl->shard_dom[std::min(k, pl->n_shards)];
        pl->shard_first[k] = D < pl->n_dom && D < (int)pl->base.size() ? pl->base[D] : pl->n_local_total;
    }
}

namespace {
ShardTable shard_table(const halo_plan* pl, const float* const* ptrs) {
    ShardTable t;
    for (int k = 0; k < kMaxShards; k++) {
        t.ptr[k] = k < pl->n_shards ? const_cast<float*>(ptrs[k]) : nullptr;
        t.first[k] = pl->shard_first[k];
    }
    return t;
}
}  // namespace

int launch_exchange_x_sharded(halo_plan* pl, float* const* shard_xyz, cudaStream_t st) {
    if (!pl->fused_ready) return HALO_EINVAL;
    if (pl->n_items_x == 0) return HALO_OK;
    XArgs a;
    a.xyz = nullptr;
    a.maps = pl->d_maps;
    a.items = pl->d_items_x;
    a.target = pl->d_target;
    a.arrived = pl->d_flags;
    a.ticket = pl->d_tickets;
    a.err = pl->d_err;
    a.n_items = pl->n_items_x;
    a.timeout_ns = pl->wait_timeout_ns;
    a.n_slots = pl->n_local_total;
    a.drop_flag = pl->drop_flag;
    a.trace = pl->trace;
    a.sh = shard_table(pl, shard_xyz);
    pl->drop_flag = -1;
    const cudaError_t e = launch_dependent(pack_x_kernel<4, true>, dim3(pl->grid_x), dim3(kThreads), st, a);
    if (e != cudaSuccess) return cuda_code(e);
    pl->launches_x++;
    return HALO_OK;
}

int launch_exchange_f_sharded(halo_plan* pl, float* const* shard_f, cudaStream_t st) {
    if (!pl->fused_ready) return HALO_EINVAL;
    if (pl->n_items_f == 0) return HALO_OK;
    const size_t nsp = (size_t)pl->n_dom * std::max(pl->P, 1);
    FArgs a;
    a.f = nullptr;
    a.pairs = pl->d_fpairs;
    a.items = pl->d_items_f;
    a.target = pl->d_target + nsp;
    a.done = pl->d_flags + nsp;
    a.ticket = pl->d_tickets + 1;
    a.err = pl->d_err;
    a.n_items = pl->n_items_f;
    a.timeout_ns = pl->wait_timeout_ns;
    a.n_slots = pl->n_local_total;
    a.trace = pl->trace ? pl->trace + 4 * (size_t)pl->n_items_x : nullptr;
    a.sh = shard_table(pl, shard_f);
    const cudaError_t e =
        launch_dependent(unpack_f_kernel<4, true>, dim3(pl->grid_f), dim3(kThreads), st, a);
    if (e != cudaSuccess) return cuda_code(e);
    pl->launches_f++;
    return HALO_OK;
}

int launch_load_home_sharded(const halo_plan* pl, const float* g, float* const* shard_local,
                             cudaStream_t st) {
    load_home_sharded_kernel<<<dim3(pl->home_grid_x, pl->n_dom), 256, 0, st>>>(
        domain_tables(pl), pl->d_home_gid, pl->n_atoms, g, shard_table(pl, shard_local), pl->n_shards,
        pl->n_local_total, pl->d_err);
    return cuda_code(cudaGetLastError());
}

int launch_store_home_sharded(const halo_plan* pl, const float* const* shard_local, float* g,
                              cudaStream_t st) {
    store_home_sharded_kernel<<<dim3(pl->home_grid_x, pl->n_dom), 256, 0, st>>>(
        domain_tables(pl), pl->d_home_gid, pl->n_atoms, shard_table(pl, shard_local), pl->n_shards, g,
        pl->n_local_total, pl->d_err);
    return cuda_code(cudaGetLastError());
}

}  // namespace halo
