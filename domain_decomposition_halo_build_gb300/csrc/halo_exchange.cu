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
// Forward progress: blocks take work items from one atomic ticket counter, in
// pulse order (ascending for coordinates, descending for forces), and a work
// item only waits on items of earlier pulses.  The earliest unfinished item was
// taken by a block that is running, and everything it waits on has an earlier
// ticket, so by induction every wait ends -- whatever the grid size and
// however the hardware schedules blocks.  Every wait is still bounded in time
// and reports HALO_ETIMEOUT through the plan's error word instead of hanging.
#include <string.h>

#include <algorithm>

#include "halo_internal.cuh"

namespace halo {
namespace {

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ int ld_relaxed_gpu(const int* p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_gpu_add(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait until *c has reached target (modulo 2^32).  On timeout the
// first waiter records where it gave up; every waiter gives up as soon as the
// plan's error word is set.
__device__ bool wait_count(const uint32_t* c, uint32_t target, int* err, long long timeout_ns,
                           int kernel, int sp, int q) {
    if ((int32_t)(ld_acquire_gpu(c) - target) >= 0) return true;
    const uint64_t t0 = global_timer_ns();
    unsigned ns = 16;
    for (;;) {
        __nanosleep(ns);
        if (ns < 256) ns <<= 1;
        if ((int32_t)(ld_acquire_gpu(c) - target) >= 0) return true;
        if (ld_relaxed_gpu(err) != 0) return false;
        if ((long long)(global_timer_ns() - t0) > timeout_ns) {
            if (atomicCAS(err, 0, HALO_ETIMEOUT) == 0) {
                err[1] = kernel;
                err[2] = sp;
                err[3] = q;
            }
            return false;
        }
    }
}

// Largest pulse q < p whose received slice (starting at oo[q]) holds local index i.
__device__ __forceinline__ int pulse_of(const int32_t* oo, int p, int i) {
    int q = p - 1;
    while (q > 0 && i < __ldg(oo + q)) q--;
    return q < 0 ? 0 : q;
}

struct XArgs {
    float* xyz;
    const int32_t* maps;
    const SPDesc* sp;
    const WorkItem* items;
    const int32_t* own_off;
    const uint32_t* nch_in;
    uint32_t* arrived;
    unsigned long long* ticket;
    int* err;
    int n_items;
    int P;
    long long timeout_ns;
    int drop_sp;
};

struct FArgs {
    float* f;
    const int32_t* maps;
    const SPDesc* sp;
    const WorkItem* items;
    const uint32_t* nch;
    const uint64_t* fmask;
    uint32_t* done;
    unsigned long long* ticket;
    int* err;
    int n_items;
    int P;
    long long timeout_ns;
};

// dst[i] = src[map[i]] + shift for i in [i0, i1).  CG: the source slots may
// have been written by other blocks of this launch, so they are read through
// L2 (ld.global.cg); otherwise they are read-only for the launch (ld.global.nc).
template <int E, bool CG>
__device__ __forceinline__ void gather_shift(const int32_t* map, const float* src, float* dst,
                                             int i0, int i1, float s0, float s1, float s2) {
    for (int b = i0; b < i1; b += kThreads * E) {
        int idx[E];
#pragma unroll
        for (int e = 0; e < E; e++) {
            const int i = b + threadIdx.x + e * kThreads;
            idx[e] = i < i1 ? __ldg(map + i) : -1;
        }
        float v[E][3];
#pragma unroll
        for (int e = 0; e < E; e++) {
            if (idx[e] >= 0) {
                const float* p = src + 3 * (int64_t)idx[e];
                if (CG) {
                    v[e][0] = __ldcg(p);
                    v[e][1] = __ldcg(p + 1);
                    v[e][2] = __ldcg(p + 2);
                } else {
                    v[e][0] = __ldg(p);
                    v[e][1] = __ldg(p + 1);
                    v[e][2] = __ldg(p + 2);
                }
            }
        }
#pragma unroll
        for (int e = 0; e < E; e++) {
            const int i = b + threadIdx.x + e * kThreads;
            if (i < i1) {
                float* q = dst + 3 * (int64_t)i;
                q[0] = v[e][0] + s0;
                q[1] = v[e][1] + s1;
                q[2] = v[e][2] + s2;
            }
        }
    }
}

template <int E>
__global__ void __launch_bounds__(kThreads) pack_x_kernel(XArgs a) {
    __shared__ int s_item;
    __shared__ uint32_t s_epoch;
    __shared__ int s_abort;
    const unsigned long long T = (unsigned long long)a.n_items + gridDim.x;
    for (;;) {
        if (threadIdx.x == 0) {
            const unsigned long long t = atomicAdd(a.ticket, 1ull);
            const unsigned long long k = t / T;
            int item = (int)(t - k * T);
            if (item < a.n_items && ld_relaxed_gpu(a.err) != 0) item = a.n_items;
            s_item = item;
            s_epoch = (uint32_t)(k + 1);
            s_abort = 0;
        }
        __syncthreads();
        const int item = s_item;
        const uint32_t epoch = s_epoch;
        if (item >= a.n_items) return;
        const WorkItem w = a.items[item];
        const SPDesc d = a.sp[w.sp];
        const int i0 = w.start, i1 = w.start + w.len;
        const int32_t* map = a.maps + d.map_off;
        const float* src = a.xyz + 3 * d.src_base;
        float* dst = a.xyz + 3 * d.dst;
        // independent entries: home atoms of the sender (Algorithm 4, first loop)
        const int ie = min(i1, d.split);
        if (i0 < ie) gather_shift<E, false>(map, src, dst, i0, ie, d.shift[0], d.shift[1], d.shift[2]);
        // dependent entries: wait for the pulses that delivered them
        if (i1 > d.split) {
            const int j0 = max(i0, d.split);
            if (threadIdx.x == 0) {
                const int32_t* oo = a.own_off + (int64_t)d.s * (a.P + 1);
                const int qlo = pulse_of(oo, d.p, __ldg(map + j0));
                const int qhi = pulse_of(oo, d.p, __ldg(map + i1 - 1));
                bool ok = true;
                for (int q = qlo; q <= qhi && ok; q++) {
                    const int sq = d.s * a.P + q;
                    ok = wait_count(a.arrived + sq, epoch * __ldg(a.nch_in + sq), a.err,
                                    a.timeout_ns, 1, w.sp, q);
                }
                s_abort = ok ? 0 : 1;
            }
            __syncthreads();
            if (s_abort) return;
            gather_shift<E, true>(map, src, dst, j0, i1, d.shift[0], d.shift[1], d.shift[2]);
        }
        // all stores of the block, then one gpu-scope release (Algorithm 5)
        __syncthreads();
        if (threadIdx.x == 0 && w.sp != a.drop_sp)
            red_release_gpu_add(a.arrived + (int64_t)d.r * a.P + d.p, 1u);
    }
}

template <int E>
__global__ void __launch_bounds__(kThreads) unpack_f_kernel(FArgs a) {
    __shared__ int s_item;
    __shared__ uint32_t s_epoch;
    __shared__ int s_abort;
    const unsigned long long T = (unsigned long long)a.n_items + gridDim.x;
    for (;;) {
        if (threadIdx.x == 0) {
            const unsigned long long t = atomicAdd(a.ticket, 1ull);
            const unsigned long long k = t / T;
            int item = (int)(t - k * T);
            if (item < a.n_items && ld_relaxed_gpu(a.err) != 0) item = a.n_items;
            s_item = item;
            s_epoch = (uint32_t)(k + 1);
            s_abort = 0;
        }
        __syncthreads();
        const int item = s_item;
        const uint32_t epoch = s_epoch;
        if (item >= a.n_items) return;
        const WorkItem w = a.items[item];
        const SPDesc d = a.sp[w.sp];
        // wait for every later pulse that writes into s's slots or into the
        // slice of r this pulse reads
        const uint64_t ms = __ldg(a.fmask + 2 * d.p), mr = __ldg(a.fmask + 2 * d.p + 1);
        if (threadIdx.x == 0 && (ms | mr)) {
            bool ok = true;
            for (uint64_t m = ms; m && ok; m &= m - 1) {
                const int q = __ffsll((long long)m) - 1;
                const int sq = d.s * a.P + q;
                ok = wait_count(a.done + sq, epoch * __ldg(a.nch + sq), a.err, a.timeout_ns, 2,
                                w.sp, q);
            }
            for (uint64_t m = mr; m && ok; m &= m - 1) {
                const int q = __ffsll((long long)m) - 1;
                const int rq = d.r * a.P + q;
                ok = wait_count(a.done + rq, epoch * __ldg(a.nch + rq), a.err, a.timeout_ns, 2,
                                w.sp, q);
            }
            s_abort = ok ? 0 : 1;
        }
        __syncthreads();
        if (s_abort) return;
        const int32_t* map = a.maps + d.map_off;
        const float* halo = a.f + 3 * d.dst;
        float* own = a.f + 3 * d.src_base;
        const int i1 = w.start + w.len;
        for (int b = w.start; b < i1; b += kThreads * E) {
            int idx[E];
#pragma unroll
            for (int e = 0; e < E; e++) {
                const int i = b + threadIdx.x + e * kThreads;
                idx[e] = i < i1 ? __ldg(map + i) : -1;
            }
            float h[E][3], o[E][3];
#pragma unroll
            for (int e = 0; e < E; e++) {
                if (idx[e] >= 0) {
                    const float* hp = halo + 3 * (int64_t)(b + threadIdx.x + e * kThreads);
                    const float* op = own + 3 * (int64_t)idx[e];
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
                if (idx[e] >= 0) {
                    float* op = own + 3 * (int64_t)idx[e];
                    op[0] = o[e][0] + h[e][0];
                    op[1] = o[e][1] + h[e][1];
                    op[2] = o[e][2] + h[e][2];
                }
            }
        }
        __syncthreads();
        if (threadIdx.x == 0) red_release_gpu_add(a.done + (int64_t)d.s * a.P + d.p, 1u);
    }
}

__global__ void load_home_kernel(const int64_t* __restrict__ home_dst,
                                 const int32_t* __restrict__ home_gid, int64_t n,
                                 const float* __restrict__ g, float* __restrict__ local) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t dd = home_dst[i], a = home_gid[i];
        local[3 * dd + 0] = g[3 * a + 0];
        local[3 * dd + 1] = g[3 * a + 1];
        local[3 * dd + 2] = g[3 * a + 2];
    }
}

__global__ void home_gid_kernel(const int64_t* __restrict__ home_dst,
                                const int32_t* __restrict__ home_gid, int64_t n,
                                int32_t* __restrict__ out) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        out[home_dst[i]] = home_gid[i];
}

// Owner id of every halo slot of one pulse (items of that pulse only).
__global__ void halo_gid_kernel(const WorkItem* __restrict__ items, const SPDesc* __restrict__ sp,
                                const int32_t* __restrict__ maps, int32_t* out) {
    const WorkItem w = items[blockIdx.x];
    const SPDesc d = sp[w.sp];
    for (int i = w.start + threadIdx.x; i < w.start + w.len; i += blockDim.x)
        out[d.dst + i] = out[d.src_base + maps[d.map_off + i]];
}

int grid_cells(const halo_plan* pl, int D, int c[3]) {
    c[0] = D % pl->grid[0];
    c[1] = (D / pl->grid[0]) % pl->grid[1];
    c[2] = D / (pl->grid[0] * pl->grid[1]);
    return 0;
}

template <class T>
int upload(T** d, const std::vector<T>& h) {
    dev_free(*d);
    HALO_TRY(dev_alloc(d, h.size()));
    if (!h.empty())
        HALO_CUDA(cudaMemcpy(*d, h.data(), h.size() * sizeof(T), cudaMemcpyHostToDevice));
    return HALO_OK;
}

template <int E>
int occupancy(int* blocks_x, int* blocks_f) {
    HALO_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_x, pack_x_kernel<E>, kThreads, 0));
    HALO_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_f, unpack_f_kernel<E>, kThreads, 0));
    return HALO_OK;
}

}  // namespace

void free_exchange(halo_plan* pl) {
    dev_free(pl->d_sp);
    dev_free(pl->d_items_x);
    dev_free(pl->d_items_f);
    dev_free(pl->d_nch);
    dev_free(pl->d_nch_in);
    dev_free(pl->d_own_off);
    dev_free(pl->d_fmask);
    dev_free(pl->d_flags);
    dev_free(pl->d_tickets);
    dev_free(pl->d_err);
}

int reset_flags(halo_plan* pl, cudaStream_t st) {
    const int nd = pl->n_dom, P = pl->P;
    if (pl->d_flags)
        HALO_CUDA(cudaMemsetAsync(pl->d_flags, 0, sizeof(uint32_t) * 2 * (size_t)nd * std::max(P, 1), st));
    if (pl->d_tickets) HALO_CUDA(cudaMemsetAsync(pl->d_tickets, 0, sizeof(unsigned long long) * 2, st));
    if (pl->d_err) HALO_CUDA(cudaMemsetAsync(pl->d_err, 0, sizeof(int) * 8, st));
    return HALO_OK;
}

int prepare_exchange(halo_plan* pl, cudaStream_t st) {
    const int nd = pl->n_dom, P = pl->P;
    // chunk size: large chunks (more independent loads per thread) when there
    // are enough of them to give every resident block several items
    const int64_t H = pl->n_halo_total;
    const int64_t resident = (int64_t)pl->num_sms * (2048 / kThreads);
    int E = 1;
    if (H / (kThreads * 4) >= 2 * resident)
        E = 4;
    else if (H / (kThreads * 2) >= resident)
        E = 2;
    pl->entries_per_thread = E;
    pl->chunk = kThreads * E;
    const int CH = pl->chunk;

    pl->sp.assign((size_t)nd * P, SPDesc{});
    std::vector<uint32_t> nch((size_t)nd * std::max(P, 1), 0), nch_in((size_t)nd * std::max(P, 1), 0);
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
            nch[sp] = (uint32_t)((x.send + CH - 1) / CH);
            nch_in[(size_t)r * P + p] = nch[sp];
        }
    }
    std::vector<WorkItem> ix, iff;
    pl->x_pulse_item_begin.assign((size_t)P + 1, 0);
    for (int p = 0; p < P; p++) {
        pl->x_pulse_item_begin[p] = (int64_t)ix.size();
        for (int s = 0; s < nd; s++) {
            const int sp = s * P + p;
            for (int st0 = 0; st0 < pl->send[sp]; st0 += CH)
                ix.push_back(WorkItem{sp, st0, std::min(CH, pl->send[sp] - st0), 0});
        }
    }
    pl->x_pulse_item_begin[P] = (int64_t)ix.size();
    for (int p = P - 1; p >= 0; p--)
        for (int s = 0; s < nd; s++) {
            const int sp = s * P + p;
            for (int st0 = 0; st0 < pl->send[sp]; st0 += CH)
                iff.push_back(WorkItem{sp, st0, std::min(CH, pl->send[sp] - st0), 0});
        }
    pl->n_items = (int)ix.size();
    // force waits: (s, p) waits for (s, q) and (r, q), q > p, whose index maps
    // can touch the same slots: pulse 0 of a later dim (its candidates include
    // every earlier slot), and, for r, the next pulse of the same dim (its
    // candidates are exactly this pulse's slice)
    std::vector<uint64_t> fmask((size_t)2 * std::max(P, 1), 0);
    for (int p = 0; p < P; p++) {
        uint64_t ms = 0, mr = 0;
        for (int q = p + 1; q < P; q++) {
            if (pl->pulse_k[q] == 0) {
                ms |= 1ull << q;
                mr |= 1ull << q;
            } else if (q == p + 1) {
                mr |= 1ull << q;
            }
        }
        fmask[2 * p] = ms;
        fmask[2 * p + 1] = mr;
    }
    HALO_TRY(upload(&pl->d_sp, pl->sp));
    HALO_TRY(upload(&pl->d_items_x, ix));
    HALO_TRY(upload(&pl->d_items_f, iff));
    HALO_TRY(upload(&pl->d_nch, nch));
    HALO_TRY(upload(&pl->d_nch_in, nch_in));
    HALO_TRY(upload(&pl->d_own_off, pl->own_off));
    HALO_TRY(upload(&pl->d_fmask, fmask));
    if (!pl->d_flags || true) {
        dev_free(pl->d_flags);
        HALO_TRY(dev_alloc(&pl->d_flags, (size_t)2 * nd * std::max(P, 1)));
    }
    if (!pl->d_tickets) HALO_TRY(dev_alloc(&pl->d_tickets, 2));
    if (!pl->d_err) HALO_TRY(dev_alloc(&pl->d_err, 8));
    int bx = 1, bf = 1;
    if (E == 4)
        HALO_TRY(occupancy<4>(&bx, &bf));
    else if (E == 2)
        HALO_TRY(occupancy<2>(&bx, &bf));
    else
        HALO_TRY(occupancy<1>(&bx, &bf));
    pl->grid_x = (int)std::min<int64_t>(pl->n_items, (int64_t)pl->num_sms * std::max(bx, 1));
    pl->grid_f = (int)std::min<int64_t>(pl->n_items, (int64_t)pl->num_sms * std::max(bf, 1));
    HALO_TRY(reset_flags(pl, st));
    return cuda_code(cudaStreamSynchronize(st));
}

int launch_exchange_x(halo_plan* pl, float* xyz, cudaStream_t st) {
    if (pl->n_items == 0) return HALO_OK;
    XArgs a;
    a.xyz = xyz;
    a.maps = pl->d_maps;
    a.sp = pl->d_sp;
    a.items = pl->d_items_x;
    a.own_off = pl->d_own_off;
    a.nch_in = pl->d_nch_in;
    a.arrived = pl->d_flags;
    a.ticket = pl->d_tickets;
    a.err = pl->d_err;
    a.n_items = pl->n_items;
    a.P = pl->P;
    a.timeout_ns = pl->wait_timeout_ns;
    a.drop_sp = pl->drop_sp;
    pl->drop_sp = -1;
    switch (pl->entries_per_thread) {
        case 4: pack_x_kernel<4><<<pl->grid_x, kThreads, 0, st>>>(a); break;
        case 2: pack_x_kernel<2><<<pl->grid_x, kThreads, 0, st>>>(a); break;
        default: pack_x_kernel<1><<<pl->grid_x, kThreads, 0, st>>>(a); break;
    }
    pl->launches_x++;
    return cuda_code(cudaGetLastError());
}

int launch_exchange_f(halo_plan* pl, float* f, cudaStream_t st) {
    if (pl->n_items == 0) return HALO_OK;
    FArgs a;
    a.f = f;
    a.maps = pl->d_maps;
    a.sp = pl->d_sp;
    a.items = pl->d_items_f;
    a.nch = pl->d_nch;
    a.fmask = pl->d_fmask;
    a.done = pl->d_flags + (size_t)pl->n_dom * pl->P;
    a.ticket = pl->d_tickets + 1;
    a.err = pl->d_err;
    a.n_items = pl->n_items;
    a.P = pl->P;
    a.timeout_ns = pl->wait_timeout_ns;
    switch (pl->entries_per_thread) {
        case 4: unpack_f_kernel<4><<<pl->grid_f, kThreads, 0, st>>>(a); break;
        case 2: unpack_f_kernel<2><<<pl->grid_f, kThreads, 0, st>>>(a); break;
        default: unpack_f_kernel<1><<<pl->grid_f, kThreads, 0, st>>>(a); break;
    }
    pl->launches_f++;
    return cuda_code(cudaGetLastError());
}

int launch_load_home(const halo_plan* pl, const float* g, float* local, cudaStream_t st) {
    const int64_t n = pl->n_atoms;
    const unsigned blocks = (unsigned)std::min<int64_t>((n + 255) / 256, (int64_t)pl->num_sms * 8);
    load_home_kernel<<<blocks, 256, 0, st>>>(pl->d_home_dst, pl->d_home_gid, n, g, local);
    return cuda_code(cudaGetLastError());
}

int launch_local_to_global(const halo_plan* pl, int32_t* out, cudaStream_t st) {
    const int64_t n = pl->n_atoms;
    const unsigned blocks = (unsigned)std::min<int64_t>((n + 255) / 256, (int64_t)pl->num_sms * 8);
    home_gid_kernel<<<blocks, 256, 0, st>>>(pl->d_home_dst, pl->d_home_gid, n, out);
    for (int p = 0; p < pl->P; p++) {
        const int64_t b = pl->x_pulse_item_begin[p], e = pl->x_pulse_item_begin[p + 1];
        if (e > b)
            halo_gid_kernel<<<(unsigned)(e - b), 256, 0, st>>>(pl->d_items_x + b, pl->d_sp,
                                                                pl->d_maps, out);
    }
    return cuda_code(cudaGetLastError());
}

}  // namespace halo
