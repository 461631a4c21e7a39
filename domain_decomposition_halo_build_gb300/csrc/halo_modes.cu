// halo_modes.cu -- three more ways to run the same exchange on one GPU.
//
// STEPWISE: one kernel launch per pulse and direction, in pulse order for
// coordinates and reverse pulse order for forces, ordered by the stream alone:
// the first fused design of the page "GPU-Initiated Halo Exchange Cuts CPU
// Bottlenecks in GROMACS" (section "Fusing pack, put, and wait into one
// kernel": one kernel per pulse, stream-ordered).
//
// STAGED: the GPU-aware-MPI schedule that page starts from (section "The CPU
// bottleneck in halo exchange"): per pulse, pulses chained Z -> Y -> X, a pack
// kernel into a send buffer, a host wait, the transfer (one kernel standing in
// for every domain's message), a host wait; forces the other way round.
//
// FLAT: because every domain lives in the same HBM, each halo slot's forwarding
// chain (page "Redesigning GROMACS Halo Exchange ...", section 3: eighth-shell
// forwarding through intermediate domains) can be composed once at build time:
//   coordinates: slot = owner's home coordinate + (L_d on every component d
//     whose chain crossed the periodic boundary) -- one fp32 add per
//     component, as in the chained exchange, because a chain crosses each
//     boundary at most once (p_d < n_d) and adds 0 to the other components;
//   forces: the copies of one owner atom form a tree (each copy's parent is the
//     slot it was received from); the chained reduction (Algorithm 6, last
//     pulse first) adds every child into its parent after the child has
//     received all of its own children, children of one parent in decreasing
//     pulse order.  Visiting an owner's copies in decreasing order of the pulse
//     that created them, and adding each into its parent, performs exactly the
//     same fp32 additions in the same order, so the results (owners and
//     intermediate halo slots) are bit-identical.
// Both passes then have no waits and no cross-block dependencies.
#include <string.h>

#include <algorithm>
#include <vector>

#include "halo_device.cuh"
#include "halo_internal.cuh"

namespace halo {
namespace {

constexpr int kNodeBits = 26;             // entry = node slot | parent position << 26
constexpr int32_t kNodeMask = (1 << kNodeBits) - 1;
constexpr int kMaxCopies = 63;            // parent positions fit in 6 bits
constexpr int kSortRegs = 8;              // copy lists sorted in registers up to this length
constexpr int32_t kXOwnerMask = (1 << 29) - 1;  // coordinate table: owner slot | crossings << 29

// A 12-byte slot as one 8-byte and one 4-byte access: the 8-byte half is
// (x, y) where the slot starts on an 8-byte boundary, else (y, z).  For the
// coordinate kernel's scattered gathers and its stores: one memory
// instruction less per slot each way (its warps stalled on a full memory
// instruction queue).  The coordinate kernel 5.91 -> 5.7 us on the 1M-atom
// system, 19.3 -> 18.6 us on the 3M.  Not for the force kernel, whose owner
// reads are coalesced across lanes: split per lane they took it from 9.6 to
// 11.3 us.
__device__ __forceinline__ void load3_nc(const float* p, float& x, float& y, float& z) {
    const bool ev = ((uintptr_t)p & 7u) == 0;
    const float2 v2 = __ldg(reinterpret_cast<const float2*>(p + (ev ? 0 : 1)));
    const float v1 = __ldg(p + (ev ? 2 : 0));
    x = ev ? v2.x : v1;
    y = ev ? v2.y : v2.x;
    z = ev ? v1 : v2.y;
}

__device__ __forceinline__ void store3(float* p, float x, float y, float z) {
    const bool ev = ((uintptr_t)p & 7u) == 0;
    *reinterpret_cast<float2*>(p + (ev ? 0 : 1)) = ev ? make_float2(x, y) : make_float2(y, z);
    p[ev ? 2 : 0] = ev ? z : x;
}

// ---- stepwise ----------------------------------------------------------------
__global__ void step_x_kernel(const SPDesc* __restrict__ sp, const int32_t* __restrict__ maps,
                              float* xyz, int P, int p, int64_t n_slots, int* err) {
    grid_launch_dependents();
    const SPDesc d = sp[(int64_t)blockIdx.y * P + p];
    const int i0 = blockIdx.x * blockDim.x + threadIdx.x;
    int m = i0 < d.send ? maps[d.map_off + i0] : 0;  // plan table: read before the wait
    grid_dependency_wait();  // pulse p - 1 (or whatever came before) has landed
    for (int i = i0; i < d.send; i += gridDim.x * blockDim.x) {
        if (i != i0) m = maps[d.map_off + i];
        if (!in_range(d.src_base + m, n_slots, err) || !in_range(d.dst + i, n_slots, err)) continue;
        const float* s = xyz + 3 * (d.src_base + m);
        float* q = xyz + 3 * (d.dst + i);
        const float v0 = s[0], v1 = s[1], v2 = s[2];
        q[0] = v0 + d.shift[0];
        q[1] = v1 + d.shift[1];
        q[2] = v2 + d.shift[2];
    }
}

__global__ void step_f_kernel(const SPDesc* __restrict__ sp, const int32_t* __restrict__ maps,
                              float* f, int P, int p, int64_t n_slots, int* err) {
    grid_launch_dependents();
    const SPDesc d = sp[(int64_t)blockIdx.y * P + p];
    const int i0 = blockIdx.x * blockDim.x + threadIdx.x;
    int m = i0 < d.send ? maps[d.map_off + i0] : 0;  // plan table: read before the wait
    grid_dependency_wait();
    for (int i = i0; i < d.send; i += gridDim.x * blockDim.x) {
        if (i != i0) m = maps[d.map_off + i];
        if (!in_range(d.src_base + m, n_slots, err) || !in_range(d.dst + i, n_slots, err)) continue;
        const float* h = f + 3 * (d.dst + i);
        float* o = f + 3 * (d.src_base + m);
        const float h0 = h[0], h1 = h[1], h2 = h[2];
        o[0] = o[0] + h0;
        o[1] = o[1] + h1;
        o[2] = o[2] + h2;
    }
}

// ---- staged (MPI-era) -----------------------------------------------------------
// Per pulse, as the GPU-aware-MPI schedule runs it: a pack kernel gathers the
// sender's entries (shifted) into a send buffer; the host waits for it; a
// transfer moves every sender's buffer slice into its receiver's halo slice
// (the MPI message; all ranks' messages of the pulse in one launch); the host
// waits for the transfer before the next pulse.  Forces run the other way,
// last pulse first: the transfer copies each receiver's halo slice into the
// buffer, the host waits, the unpack kernel adds it into the sender's mapped
// slots, the host waits.  The buffer slice of (s, p) sits at the map's own
// offset (the maps tile the halo slots pulse by pulse), so the buffer has one
// 12-byte element per halo slot.
__global__ void staged_pack_x_kernel(const SPDesc* __restrict__ sp, const int32_t* __restrict__ maps,
                                     const float* __restrict__ xyz, float* __restrict__ buf, int P,
                                     int p, int64_t n_slots, int64_t n_buf, int* err) {
    const SPDesc d = sp[(int64_t)blockIdx.y * P + p];
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < d.send; i += gridDim.x * blockDim.x) {
        const int64_t m = d.src_base + maps[d.map_off + i];
        if (!in_range(m, n_slots, err) || !in_range(d.map_off + i, n_buf, err)) continue;
        const float* s = xyz + 3 * m;
        float* b = buf + 3 * (d.map_off + i);
        b[0] = s[0] + d.shift[0];
        b[1] = s[1] + d.shift[1];
        b[2] = s[2] + d.shift[2];
    }
}

// TO_HALO: buffer slice -> receiver's halo slice (coordinates); else the
// halo slice -> buffer slice (forces).
template <bool TO_HALO>
__global__ void staged_move_kernel(const SPDesc* __restrict__ sp, float* local, float* buf, int P, int p,
                                   int64_t n_slots, int64_t n_buf, int* err) {
    const SPDesc d = sp[(int64_t)blockIdx.y * P + p];
    const int n = 3 * d.send;
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < n; j += gridDim.x * blockDim.x) {
        if (!in_range(d.dst + j / 3, n_slots, err) || !in_range(d.map_off + j / 3, n_buf, err)) continue;
        if (TO_HALO)
            local[3 * d.dst + j] = buf[3 * d.map_off + j];
        else
            buf[3 * d.map_off + j] = local[3 * d.dst + j];
    }
}

__global__ void staged_unpack_f_kernel(const SPDesc* __restrict__ sp, const int32_t* __restrict__ maps,
                                       float* f, const float* __restrict__ buf, int P, int p,
                                       int64_t n_slots, int64_t n_buf, int* err) {
    const SPDesc d = sp[(int64_t)blockIdx.y * P + p];
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < d.send; i += gridDim.x * blockDim.x) {
        const int64_t m = d.src_base + maps[d.map_off + i];
        if (!in_range(m, n_slots, err) || !in_range(d.map_off + i, n_buf, err)) continue;
        const float* h = buf + 3 * (d.map_off + i);
        float* o = f + 3 * m;
        const float h0 = h[0], h1 = h[1], h2 = h[2];
        o[0] = o[0] + h0;
        o[1] = o[1] + h1;
        o[2] = o[2] + h2;
    }
}

// ---- flat: build-time composition of the chains -------------------------------

// Pulse p, in ascending order: every received slot inherits its source's owner
// and boundary crossings, and remembers its source (parent) and pulse.  It
// also writes its coordinate-table entry (owner | crossings << 29, at
// xbase[receiver] + slot) and counts its owner's copies, keeping its rank
// among them (the counter's value before its increment).
__global__ void chain_pulse_kernel(const SPDesc* __restrict__ sp, const int32_t* __restrict__ maps,
                                   int32_t* owner, int32_t* parent, int8_t* hop, int8_t* code,
                                   const int32_t* __restrict__ xbase, int32_t* __restrict__ xflat,
                                   int32_t* ncopies, int32_t* __restrict__ rank, int P, int p,
                                   int dim) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    const SPDesc d = sp[(int64_t)blockIdx.y * P + p];
    if (d.send <= 0) return;
    const int8_t bit = d.shift[dim] != 0.0f ? (int8_t)(1 << dim) : (int8_t)0;
    const int64_t xb = xbase[d.r];
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < d.send; i += gridDim.x * blockDim.x) {
        const int64_t h = d.dst + i;
        const int64_t src = d.src_base + maps[d.map_off + i];
        // entries below the split are home slots: their own owner, no
        // crossings; the rest were received (and filled) in earlier pulses.
        // Home slots' entries of these arrays are never read, so nothing
        // initialises them.
        const bool home = i < d.split;
        const int32_t o = home ? (int32_t)src : owner[src];
        const int8_t c = (int8_t)((home ? 0 : code[src]) | bit);
        owner[h] = o;
        parent[h] = (int32_t)src;
        hop[h] = (int8_t)p;
        code[h] = c;
        xflat[xb + h] = o | ((int32_t)c << 29);
        rank[h] = atomicAdd(ncopies + o, 1);
    }
}

// The coordinate kernel's work items: domain D's halo range in chunks of
// `chunk` slots, numbered in domain order; item b = {b * chunk (its table
// offset), first halo slot, count}; xbase[D] = the table offset of D's halo
// slot 0 minus the slot (halo slot h of D sits at xbase[D] + h).  Block g
// takes domains [32g, 32g + 32): it sums the item counts of the domains
// before them (every block for itself: a few hundred L2 loads), warp 0 scans
// its 32, and warp w writes domain 32g + w's items.
__global__ void __launch_bounds__(1024) xflat_items_kernel(DomainTables t, int nd, int P, int chunk,
                                                           int4* __restrict__ items,
                                                           int32_t* __restrict__ xbase) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    __shared__ int64_t sfirst[32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g0 = blockIdx.x * 32;
    auto count = [&](int D) -> int64_t {
        const int64_t nh = t.own_off[(int64_t)D * (P + 1) + P] - t.n_home[D];
        return (nh + chunk - 1) / chunk;
    };
    int64_t carry = 0;
    for (int D0 = 0; D0 < g0; D0 += 1024) {
        const int D = D0 + threadIdx.x;
        int64_t tot;
        block_exclusive_scan<1024>(D < g0 ? count(D) : 0, &tot);
        carry += tot;
    }
    if (warp == 0) {
        const int D = g0 + lane;
        const int64_t c = D < nd ? count(D) : 0;
        int64_t x = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x += y;
        }
        sfirst[lane] = carry + x - c;
    }
    __syncthreads();
    const int D = g0 + warp;
    if (D >= nd) return;
    const int64_t nh = t.own_off[(int64_t)D * (P + 1) + P] - t.n_home[D];
    const int64_t d0 = t.base[D] + t.n_home[D];
    const int64_t f = sfirst[warp];
    if (lane == 0) xbase[D] = (int32_t)(f * chunk - d0);  // table offset - first halo slot
    for (int64_t k = lane; k * chunk < nh; k += 32) {
        const int64_t b = f + k;
        items[b] = make_int4((int)(b * chunk), (int)(d0 + k * chunk), (int)min((int64_t)chunk, nh - k * chunk), 0);
    }
}

// Two exclusive scans in one pass over an int32 array: channel a in the low
// 32 bits of an int64, channel b in the high 32 bits (no carry: every prefix
// of a stays below 2^32).  SRC 0, over local slots: a = copies of the slot,
// b = 1 if it has any (an owner).  SRC 1, over owners: a = 1 for a class-A
// tree (<= 3 copies), b = 1 for class B (4..11 copies), from the entry
// offsets (element i reads in[i] and in[i + 1]).
template <int SRC>
__device__ __forceinline__ int64_t pair_value(const int32_t* __restrict__ in, int64_t i) {
    if (SRC == 0) {
        const int32_t v = in[i];
        return (int64_t)v | ((int64_t)(v > 0 ? 1 : 0) << 32);
    }
    const int32_t k = in[i + 1] - in[i];
    return (int64_t)(k <= 3 ? 1 : 0) | ((int64_t)(k > 3 && k <= 11 ? 1 : 0) << 32);
}

// The element count n comes from the host, or (n_dev != nullptr) from the
// device: the high half of *n_dev (the owner count of the SRC 0 scan's grand
// total), with the grid sized for the host bound n.
__device__ __forceinline__ int64_t scan_count(int64_t n, const int64_t* n_dev) {
    return n_dev ? (*n_dev >> 32) : n;
}

// Elements i .. i + 7 of a pair scan (pair_value), 0 past n; i is a multiple
// of 8 and `in` 16-byte aligned, so a whole group is two 16-byte loads (SRC 1
// also reads in[i + 8]).
template <int SRC>
__device__ __forceinline__ void pair_load8(const int32_t* __restrict__ in, int64_t i, int64_t n,
                                           int64_t v[8]) {
    if (i + 8 <= n) {
        const int4 x0 = *reinterpret_cast<const int4*>(in + i);
        const int4 x1 = *reinterpret_cast<const int4*>(in + i + 4);
        const int32_t e[9] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w, SRC == 1 ? in[i + 8] : 0};
#pragma unroll
        for (int k = 0; k < 8; k++) {
            if (SRC == 0) {
                v[k] = (int64_t)e[k] | ((int64_t)(e[k] > 0 ? 1 : 0) << 32);
            } else {
                const int32_t c = e[k + 1] - e[k];
                v[k] = (int64_t)(c <= 3 ? 1 : 0) | ((int64_t)(c > 3 && c <= 11 ? 1 : 0) << 32);
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; k++) v[k] = i + k < n ? pair_value<SRC>(in, i + k) : 0;
    }
}

// Tile sums: thread t of block b sums elements b * kScanTile + 8t .. + 7.
template <int SRC>
__global__ void __launch_bounds__(kThreads) pair_reduce_kernel(const int32_t* __restrict__ in,
                                                               int64_t n, const int64_t* n_dev,
                                                               int64_t* __restrict__ sums) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    static_assert(kScanTile == 8 * kThreads, "eight elements per thread");
    __shared__ int64_t ws[kThreads / 32];
    n = scan_count(n, n_dev);
    const int64_t b0 = (int64_t)blockIdx.x * kScanTile;
    if (b0 >= n) return;
    int64_t v[8];
    pair_load8<SRC>(in, b0 + 8 * threadIdx.x, n, v);
    int64_t s = 0;
#pragma unroll
    for (int k = 0; k < 8; k++) s += v[k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
    if ((threadIdx.x & 31) == 0) ws[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        int64_t t = 0;
        for (int w = 0; w < kThreads / 32; w++) t += ws[w];
        sums[blockIdx.x] = t;
    }
}

// Scans the nb tile sums in place and stores the grand total in sums[nb]
// and, if given, in *total.  end (SRC 0): the owner list's end offset,
// end[owners] = copies.
__global__ void __launch_bounds__(1024) pair_top_kernel(int64_t* __restrict__ sums, int64_t n,
                                                        const int64_t* n_dev, int64_t* total,
                                                        int32_t* end) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    n = scan_count(n, n_dev);
    const int64_t nb = (n + kScanTile - 1) / kScanTile;
    int64_t carry = 0;
    for (int64_t b = 0; b < nb; b += 1024) {
        const int64_t i = b + threadIdx.x;
        const int64_t v = i < nb ? sums[i] : 0;
        int64_t tot;
        const int64_t pre = block_exclusive_scan<1024>(v, &tot);
        if (i < nb) sums[i] = carry + pre;
        carry += tot;
    }
    if (threadIdx.x == 0) {
        sums[nb] = carry;
        if (total) *total = carry;
        if (end) end[carry >> 32] = (int32_t)(carry & 0xffffffffll);
    }
}

// Down pass: thread t of block b takes elements b * kScanTile + 8t .. + 7
// (two 16-byte loads), one block scan of the thread sums gives its first
// prefix, and it writes its eight exclusive prefixes.  SRC 0 also writes the
// owner list: for a slot with copies, fown[its owner index] = the slot and
// fstart[...] = its first entry (out_b, the owner indices, is then not
// stored), through shared memory.
template <int SRC>
__global__ void __launch_bounds__(kThreads) pair_down_kernel(const int32_t* __restrict__ in, int64_t n,
                                                             const int64_t* n_dev,
                                                             const int64_t* __restrict__ sums,
                                                             int32_t* __restrict__ out_a,
                                                             int32_t* __restrict__ out_b,
                                                             int32_t* __restrict__ fown,
                                                             int32_t* __restrict__ fstart) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    n = scan_count(n, n_dev);
    const int64_t b0 = (int64_t)blockIdx.x * kScanTile;
    if (b0 >= n) return;
    const int64_t i0 = b0 + 8 * threadIdx.x;
    int64_t v[8];
    pair_load8<SRC>(in, i0, n, v);
    int64_t t = 0;
#pragma unroll
    for (int k = 0; k < 8; k++) t += v[k];
    int64_t tot;
    const int64_t first = sums[blockIdx.x];
    int64_t run = first + block_exclusive_scan<kThreads>(t, &tot);
    // SRC 0: the block's owners take the contiguous owner indices from
    // first >> 32 on; they are staged in shared memory and written out
    // coalesced
    __shared__ int32_t s_own[SRC == 0 ? kScanTile : 1], s_start[SRC == 0 ? kScanTile : 1];
    const int32_t own0 = (int32_t)(first >> 32);
    int32_t a[8], bb[8];
#pragma unroll
    for (int k = 0; k < 8; k++) {
        a[k] = (int32_t)(run & 0xffffffffll);
        bb[k] = (int32_t)(run >> 32);
        if (SRC == 0 && fown && (v[k] & 0xffffffffll) > 0 && i0 + k < n) {
            s_own[bb[k] - own0] = (int32_t)(i0 + k);
            s_start[bb[k] - own0] = a[k];
        }
        run += v[k];
    }
    if (SRC == 0 && fown) {
        __syncthreads();
        const int n_own = (int)(tot >> 32);  // owners in this block's tile
        for (int j = threadIdx.x; j < n_own; j += kThreads) {
            fown[own0 + j] = s_own[j];
            fstart[own0 + j] = s_start[j];
        }
    }
    const bool write_b = !(SRC == 0 && fown);
    if (i0 + 8 <= n) {
        *reinterpret_cast<int4*>(out_a + i0) = make_int4(a[0], a[1], a[2], a[3]);
        *reinterpret_cast<int4*>(out_a + i0 + 4) = make_int4(a[4], a[5], a[6], a[7]);
        if (write_b) {
            *reinterpret_cast<int4*>(out_b + i0) = make_int4(bb[0], bb[1], bb[2], bb[3]);
            *reinterpret_cast<int4*>(out_b + i0 + 4) = make_int4(bb[4], bb[5], bb[6], bb[7]);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; k++) {
            if (i0 + k < n) {
                out_a[i0 + k] = a[k];
                if (write_b) out_b[i0 + k] = bb[k];
            }
        }
    }
}

// Launches the three passes; sums holds ceil(n / kScanTile) + 1 int64 (the
// grand total lands in its last entry, and in *total if given).  n_dev: see
// scan_count (n is then the bound the grids are sized for).
template <int SRC>
int pair_scan(const int32_t* in, int64_t n, const int64_t* n_dev, int64_t* sums, int32_t* out_a,
              int32_t* out_b, int64_t* total, cudaStream_t st, int32_t* fown = nullptr,
              int32_t* fstart = nullptr) {
    const int64_t nb = (n + kScanTile - 1) / kScanTile;
    if (nb > 0)
        HALO_CUDA(launch_dependent_shm(pair_reduce_kernel<SRC>, dim3((unsigned)nb), dim3(kThreads), 0, st,
                                       in, n, n_dev, sums));
    HALO_CUDA(launch_dependent_shm(pair_top_kernel, dim3(1), dim3(1024), 0, st, sums, n, n_dev, total,
                                   fstart));
    if (nb > 0)
        HALO_CUDA(launch_dependent_shm(pair_down_kernel<SRC>, dim3((unsigned)nb), dim3(kThreads), 0, st,
                                       in, n, n_dev, (const int64_t*)sums, out_a, out_b, fown, fstart));
    return HALO_OK;
}

// Every halo slot into its owner's copy list, at the rank chain_pulse_kernel
// took.  The blocks stride over the coordinate items (a block per item
// would launch one short block per 256-384 slots).
__global__ void owner_fill_kernel(const int4* __restrict__ items, int n_items,
                                  const int32_t* __restrict__ owner,
                                  const int32_t* __restrict__ entry_pos,
                                  const int32_t* __restrict__ rank, int32_t* __restrict__ tmp) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    for (int b = blockIdx.x; b < n_items; b += gridDim.x) {
        const int4 it = items[b];
        for (int i = threadIdx.x; i < it.z; i += blockDim.x) {
            const int64_t j = (int64_t)it.y + i;
            tmp[entry_pos[owner[j]] + rank[j]] = (int32_t)j;
        }
    }
}

// Owner records (the force pass's tables): class A -- up to 3 copies, one
// 16-byte record {home | k << 26, three entries}; class B -- up to 11 copies,
// three 16-byte records; class C -- more copies, {header, first entry} into
// the entry list.  An entry is node slot | parent position << 26.
__device__ __forceinline__ void write_rec_a(int4* recA, int32_t hdr, const int32_t* e, int k) {
    *recA = make_int4(hdr, e[0], k > 1 ? e[1] : 0, k > 2 ? e[2] : 0);
}

template <int N>
__device__ __forceinline__ void write_rec_b(int4* recB, int32_t hdr, const int32_t (&e)[N], int k) {
    int32_t w[11];
#pragma unroll
    for (int j = 0; j < 11; j++) w[j] = j < k && j < N ? e[j] : 0;
    recB[0] = make_int4(hdr, w[0], w[1], w[2]);
    recB[1] = make_int4(w[3], w[4], w[5], w[6]);
    recB[2] = make_int4(w[7], w[8], w[9], w[10]);
}

// Per owner: order its copies by decreasing creating pulse (ties by slot),
// replace each copy's parent slot by the parent's position (0 = the owner),
// and write the owner's record at its class position (posA / posB from the
// class scan; class C after them, with its entries in the entry list).
// Owners of up to three copies (class A, nearly all) are done here; the
// others are listed (listB[posB[m]], listC[class-C rank]) for
// owner_sort_bc_kernel, so that no warp here runs the longer sorts.
__global__ void owner_sort_kernel(const int32_t* __restrict__ fown, const int32_t* __restrict__ fstart,
                                  const int32_t* __restrict__ tmp, const int32_t* __restrict__ parent,
                                  const int8_t* __restrict__ hop, const int64_t* __restrict__ total,
                                  const int32_t* __restrict__ posA, const int32_t* __restrict__ posB,
                                  int4* __restrict__ recA, int32_t* __restrict__ listB,
                                  int32_t* __restrict__ listC, int* max_copies, int* err) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    const int64_t n_owners = *total >> 32;
    __shared__ int block_max;
    if (threadIdx.x == 0) block_max = 0;
    __syncthreads();
    int my_max = 0;
    for (int64_t m = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; m < n_owners;
         m += (int64_t)gridDim.x * blockDim.x) {
        const int s0 = fstart[m], k = fstart[m + 1] - s0;
        my_max = max(my_max, k);
        if (k > kMaxCopies) atomicCAS(err, 0, HALO_ECAPACITY);  // listed below, skipped there
        const int32_t hdr = fown[m] | (k << kNodeBits);
        if (k == 1) {  // most owners: a single copy, received from the owner itself
            const int32_t v = tmp[s0];
            if (parent[v] != fown[m]) atomicCAS(err, 0, HALO_ECAPACITY);
            recA[posA[m]] = make_int4(hdr, v, 0, 0);
            continue;
        }
        if (k <= 3) {
            // two or three copies (most multi-copy owners): three compare-
            // exchanges on (pulse descending, slot ascending)
            int32_t nd3[3];
            int hp3[3];
#pragma unroll
            for (int j = 0; j < 3; j++) {
                nd3[j] = j < k ? tmp[s0 + j] : INT32_MAX;
                hp3[j] = j < k ? (int)hop[nd3[j]] : -1000;
            }
            auto cx = [&](int a, int b) {
                const bool swap = hp3[a] < hp3[b] || (hp3[a] == hp3[b] && nd3[a] > nd3[b]);
                if (swap) {
                    const int32_t tn = nd3[a];
                    nd3[a] = nd3[b];
                    nd3[b] = tn;
                    const int th = hp3[a];
                    hp3[a] = hp3[b];
                    hp3[b] = th;
                }
            };
            cx(0, 1);
            cx(1, 2);
            cx(0, 1);
            const int32_t home = fown[m];
            int32_t e3[3] = {0, 0, 0};
#pragma unroll
            for (int j = 0; j < 3; j++) {
                if (j < k) {
                    const int32_t ps = parent[nd3[j]];
                    int pos = 0;
                    if (ps != home) {
#pragma unroll
                        for (int q = 2; q > j; q--)
                            if (q < k && nd3[q] == ps) pos = q + 1;
                        if (pos == 0) atomicCAS(err, 0, HALO_ECAPACITY);  // parent not among the copies
                    }
                    e3[j] = nd3[j] | (pos << kNodeBits);
                }
            }
            write_rec_a(recA + posA[m], hdr, e3, k);
            continue;
        }
        if (k <= 11)
            listB[posB[m]] = (int32_t)m;
        else
            listC[m - posA[m] - posB[m]] = (int32_t)m;  // class-C owners before m
    }
    atomicMax(&block_max, my_max);
    __syncthreads();
    if (threadIdx.x == 0) atomicMax(max_copies, block_max);
}

// The owners of four or more copies (classes B and C), from the lists
// owner_sort_kernel wrote: counts[0] = copies | owners << 32, counts[1] =
// class A | class B << 32.  If host_out is given (the host's mapped
// staging), the last block to finish (ticket in misc[2]) copies the build's
// summary words misc[0 .. 11] there.
__global__ void owner_sort_bc_kernel(const int32_t* __restrict__ fown, const int32_t* __restrict__ fstart,
                                     const int32_t* __restrict__ tmp, const int32_t* __restrict__ parent,
                                     const int8_t* __restrict__ hop, const int64_t* __restrict__ counts,
                                     const int32_t* __restrict__ posA, const int32_t* __restrict__ posB,
                                     const int32_t* __restrict__ listB, const int32_t* __restrict__ listC,
                                     int4* __restrict__ recB, int4* __restrict__ recC,
                                     int32_t* __restrict__ fent, int* err, int32_t* misc,
                                     int32_t* __restrict__ host_out) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    const int64_t n_owners = counts[0] >> 32;
    const int64_t n_a = counts[1] & 0xffffffffll, n_b = counts[1] >> 32;
    const int64_t n_bc = n_owners - n_a;
    for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n_bc;
         q += (int64_t)gridDim.x * blockDim.x) {
        const int64_t m = q < n_b ? listB[q] : listC[q - n_b];
        const int s0 = fstart[m], k = fstart[m + 1] - s0;
        if (k > kMaxCopies) continue;  // reported by owner_sort_kernel
        const int32_t hdr = fown[m] | (k << kNodeBits);
        if (k <= kSortRegs) {
            // the same order in registers: a fully unrolled exchange sort on
            // (pulse descending, slot ascending); unused places sort last
            int32_t nd8[kSortRegs];
            int hp8[kSortRegs];
#pragma unroll
            for (int j = 0; j < kSortRegs; j++) {
                nd8[j] = j < k ? tmp[s0 + j] : INT32_MAX;
                hp8[j] = j < k ? (int)hop[nd8[j]] : -1000;
            }
#pragma unroll
            for (int a = 0; a < kSortRegs - 1; a++)
#pragma unroll
                for (int b = 0; b < kSortRegs - 1 - a; b++) {
                    const bool swap = hp8[b] < hp8[b + 1] || (hp8[b] == hp8[b + 1] && nd8[b] > nd8[b + 1]);
                    if (swap) {
                        const int32_t tn = nd8[b];
                        nd8[b] = nd8[b + 1];
                        nd8[b + 1] = tn;
                        const int th = hp8[b];
                        hp8[b] = hp8[b + 1];
                        hp8[b + 1] = th;
                    }
                }
            const int32_t home = fown[m];
            int32_t e8[kSortRegs];
#pragma unroll
            for (int j = 0; j < kSortRegs; j++) {
                e8[j] = 0;
                if (j < k) {
                    const int32_t ps = parent[nd8[j]];
                    int pos = 0;
                    if (ps != home) {
#pragma unroll
                        for (int q = kSortRegs - 1; q > j; q--)
                            if (q < k && nd8[q] == ps) pos = q + 1;
                        if (pos == 0) atomicCAS(err, 0, HALO_ECAPACITY);  // parent not among the copies
                    }
                    e8[j] = nd8[j] | (pos << kNodeBits);
                }
            }
            write_rec_b(recB + 3 * (int64_t)posB[m], hdr, e8, k);  // 4..8 copies: class B
            continue;
        }
        int32_t node[kMaxCopies];
        int8_t hp[kMaxCopies];
        for (int j = 0; j < k; j++) {
            const int32_t v = tmp[s0 + j];
            int8_t hv = hop[v];
            int i = j;
            while (i > 0 && (hp[i - 1] < hv || (hp[i - 1] == hv && node[i - 1] > v))) {
                node[i] = node[i - 1];
                hp[i] = hp[i - 1];
                i--;
            }
            node[i] = v;
            hp[i] = hv;
        }
        const int32_t home = fown[m];
        for (int j = 0; j < k; j++) {
            const int32_t ps = parent[node[j]];
            int pos = 0;
            if (ps != home) {
                for (int q = j + 1; q < k; q++)
                    if (node[q] == ps) {
                        pos = q + 1;
                        break;
                    }
                if (pos == 0) atomicCAS(err, 0, HALO_ECAPACITY);  // parent not among the copies
            }
            node[j] = node[j] | (pos << kNodeBits);  // the entry, in place
        }
        if (k <= 11) {
            int32_t e11[11];
            for (int j = 0; j < 11; j++) e11[j] = j < k ? node[j] : 0;
            write_rec_b(recB + 3 * (int64_t)posB[m], hdr, e11, k);
        } else {
            for (int j = 0; j < k; j++) fent[s0 + j] = node[j];
            recC[m - posA[m] - posB[m]] = make_int4(hdr, s0, 0, 0);  // class-C owners before m
        }
    }
    if (host_out) {
        __shared__ int last;
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) last = atomicAdd(misc + 2, 1) == (int)gridDim.x - 1;
        __syncthreads();
        if (last) {
            __threadfence();
            if (threadIdx.x < 12) host_out[threadIdx.x] = __ldcg(misc + threadIdx.x);
        }
    }
}

// ---- flat: the exchanges ------------------------------------------------------------
// Plan tables of the block that will take this block's place when it exits
// (blockIdx.x + ahead, ahead = the resident blocks of the launch), into L2:
// that block's first dependent round trip then comes from L2.  A grid of
// more than one wave gains: x + f 18.45 -> 18.18 us on the 1M-atom system,
// 54.2 -> 52.7 us on the 3M.
__device__ __forceinline__ void prefetch_table(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// Threads per block of the coordinate kernel.  128 rather than 256: twice the
// blocks spread more evenly over the SMs, and as they finish they free room
// sooner for the next kernel's blocks (programmatic dependent launch).  On
// the 1M-atom system x + f back to back took 18.4 us instead of 19.5.
constexpr int kXT = 128;
template <int E>
__global__ void __launch_bounds__(kXT) flat_x_kernel(float* xyz, const int32_t* __restrict__ xflat,
                                                     const int4* __restrict__ items, float L0, float L1,
                                                     float L2, int64_t n_slots, int* err, int ahead) {
    grid_launch_dependents();
    if (ahead > 0 && blockIdx.x + ahead < gridDim.x) {
#pragma unroll
        for (int e = 0; e < E; e++)
            prefetch_table(xflat + (int64_t)(blockIdx.x + ahead) * (kXT * E) + threadIdx.x + e * kXT);
        if (threadIdx.x == 0) prefetch_table(items + blockIdx.x + ahead);
    }
    // block b's table entries start at b * kXT * E (the table is padded per
    // chunk), so they load alongside the item instead of after it; entries
    // at or past the item's count are padding and never used
    int32_t v[E];
#pragma unroll
    for (int e = 0; e < E; e++)
        v[e] = __ldg(xflat + (int64_t)blockIdx.x * (kXT * E) + threadIdx.x + e * kXT);
    int4 it = items[blockIdx.x];
    if (!in_range((int64_t)it.y + it.z - 1, n_slots, err)) it.z = 0;
    // Blocks of the first wave (the only ones that can start before the
    // kernel ahead has finished) warm their gather lines in L2 meanwhile.
    // L2 is the device's point of coherence: a prefetch hands no thread a
    // value, so it cannot expose anything older than the preceding grid's
    // writes.  1M-atom system, x + f back to back: 17.2 -> 15.8 us.
    if (blockIdx.x < ahead) {
#pragma unroll
        for (int e = 0; e < E; e++)
            if (threadIdx.x + e * kXT < it.z) prefetch_table(xyz + 3 * (int64_t)(v[e] & kXOwnerMask));
    }
    // the chunk and its codes are plan tables; coordinates only after the wait
    grid_dependency_wait();
    float a[E][3];
#pragma unroll
    for (int e = 0; e < E; e++) {
        if (threadIdx.x + e * kXT < it.z) {
            // owners are home slots, never written by this kernel
            const int64_t o = v[e] & kXOwnerMask;
            const float* s = xyz + 3 * (in_range(o, n_slots, err) ? o : 0);
            load3_nc(s, a[e][0], a[e][1], a[e][2]);
        }
    }
    if (E < 3) {
        // small chunks (two slots per thread): direct stores, where a bulk
        // copy's round trip does not pay
#pragma unroll
        for (int e = 0; e < E; e++) {
            const int i = threadIdx.x + e * kXT;
            if (i < it.z) {
                const unsigned c = (unsigned)v[e] >> 29;
                float* q = xyz + 3 * ((int64_t)it.y + i);
                store3(q, a[e][0] + ((c & 1u) ? L0 : 0.0f), a[e][1] + ((c & 2u) ? L1 : 0.0f),
                       a[e][2] + ((c & 4u) ? L2 : 0.0f));
            }
        }
        return;
    }
    // the chunk's halo slots are contiguous: stage them, one bulk copy out
    __shared__ __align__(128) float stage[3 * kXT * E + 4];
    float* dst = xyz + 3 * (int64_t)it.y;
    const int sh = stage_shift(dst);
#pragma unroll
    for (int e = 0; e < E; e++) {
        const int i = threadIdx.x + e * kXT;
        if (i < it.z) {
            const unsigned c = (unsigned)v[e] >> 29;
            float* q = stage + sh + 3 * i;
            q[0] = a[e][0] + ((c & 1u) ? L0 : 0.0f);
            q[1] = a[e][1] + ((c & 2u) ? L1 : 0.0f);
            q[2] = a[e][2] + ((c & 4u) ? L2 : 0.0f);
        }
    }
    fence_smem_to_async();
    __syncthreads();
    if (threadIdx.x == 0) bulk_store_floats(dst, stage, 3 * it.z, false);
}

// Reduction of N owners' copy trees held in registers (k <= K copies each).
// All loads of the N trees are issued before any arithmetic (their slots never
// overlap, which the compiler cannot know), so a thread keeps N trees' worth of
// loads in flight.  Copy q receives its children (all earlier in the order) in
// ascending position, then the owner receives its children: every accumulator
// sees the same adds in the same order as the chained reduction.
struct NoMid {
    __device__ void operator()() const {}
};

template <int K, int N, class Mid = NoMid>
__device__ __forceinline__ void reduce_trees(float* f, const int32_t (&home)[N], const int (&kk)[N],
                                             const int32_t (&ent)[N][K], Mid mid = Mid()) {
    float c0[N][3], c[N][K][3];
    int par[N][K];
#pragma unroll
    for (int o = 0; o < N; o++) {
        if (kk[o] > 0) {
            const float* fh = f + 3 * (int64_t)home[o];
            c0[o][0] = fh[0];
            c0[o][1] = fh[1];
            c0[o][2] = fh[2];
        }
#pragma unroll
        for (int j = 0; j < K; j++) {
            par[o][j] = -1;
            if (j < kk[o]) {
                const float* fn = f + 3 * (int64_t)(ent[o][j] & kNodeMask);
                c[o][j][0] = fn[0];
                c[o][j][1] = fn[1];
                c[o][j][2] = fn[2];
                par[o][j] = (int)((unsigned)ent[o][j] >> kNodeBits);
            }
        }
    }
    mid();  // runs while this thread's loads are in flight
#pragma unroll
    for (int o = 0; o < N; o++) {
        if (kk[o] <= 0) continue;
        unsigned has_child = 0;
#pragma unroll
        for (int q = 1; q < K; q++) {
#pragma unroll
            for (int j = 0; j < q; j++) {
                if (par[o][j] == q + 1) {
                    c[o][q][0] = c[o][q][0] + c[o][j][0];
                    c[o][q][1] = c[o][q][1] + c[o][j][1];
                    c[o][q][2] = c[o][q][2] + c[o][j][2];
                    has_child |= 1u << q;
                }
            }
        }
#pragma unroll
        for (int j = 0; j < K; j++) {
            if (par[o][j] == 0) {
                c0[o][0] = c0[o][0] + c[o][j][0];
                c0[o][1] = c0[o][1] + c[o][j][1];
                c0[o][2] = c0[o][2] + c[o][j][2];
            }
        }
        float* fh = f + 3 * (int64_t)home[o];
        fh[0] = c0[o][0];
        fh[1] = c0[o][1];
        fh[2] = c0[o][2];
#pragma unroll
        for (int j = 0; j < K; j++) {
            if (has_child >> j & 1u) {
                float* fn = f + 3 * (int64_t)(ent[o][j] & kNodeMask);
                fn[0] = c[o][j][0];
                fn[1] = c[o][j][1];
                fn[2] = c[o][j][2];
            }
        }
    }
}

template <int K>
__device__ __forceinline__ void reduce_tree(float* f, int32_t home, int k, const int32_t (&ent)[K]) {
    const int32_t h[1] = {home};
    const int kk[1] = {k};
    int32_t e[1][K];
#pragma unroll
    for (int j = 0; j < K; j++) e[0][j] = ent[j];
    reduce_trees<K, 1>(f, h, kk, e);
}

// One thread per owner with copies.  Owners come in three record classes
// (sorted by class, then by home slot): A -- up to 3 copies, one 16-byte
// record {home | k << 26, three entries}; B -- up to 11 copies, three 16-byte
// records; C -- more copies, {header, first entry} into the entry list.  A
// record is one load, so the forces follow after a single dependent round
// trip.  KB: copies held in registers for class B (7 or 11, the plan's
// largest tree); KW: class C trees of up to KW copies in registers (0: none),
// larger ones reduced sequentially through memory in the same order.
// Debug builds: a tree whose home slot, node slots or parent positions fall
// outside their ranges is skipped (0 copies) and HALO_EBOUNDS recorded.
template <int K>
__device__ __forceinline__ int checked_copies(int32_t home, int k, const int32_t (&ent)[K],
                                              int64_t n_slots, int* err) {
#ifdef HALO_DEBUG
    bool ok = k <= K && in_range(home, n_slots, err);
#pragma unroll
    for (int j = 0; j < K; j++)
        if (j < k)
            ok = ok && in_range(ent[j] & kNodeMask, n_slots, err) &&
                 in_range((unsigned)ent[j] >> kNodeBits, k + 1, err);
    return ok ? k : 0;
#else
    return k;
#endif
}

// class-A owners per thread: a tile is kFlatA * kThreads owners (at 2 the
// kernel fits four blocks per SM; 3 and 4 owners needed 80 and 114 registers
// and fit fewer blocks)
constexpr int kFlatA = 2;

template <int KB, int KW>
__global__ void __launch_bounds__(kThreads) flat_f_kernel(float* f, const int4* __restrict__ recA,
                                                          int64_t nA, const int4* __restrict__ recB,
                                                          int64_t nB, const int4* __restrict__ recC,
                                                          int64_t nC, const int32_t* __restrict__ fent,
                                                          int64_t n_slots, int64_t n_fent, int* err,
                                                          int64_t ahead) {
    // blocks [0, tilesBC) take classes B and C, one owner per thread (the
    // longer trees start first); the following blocks take class-A tiles of
    // kFlatA * blockDim owners, kFlatA per thread (coalesced record loads), so
    // both kinds of trees run side by side
    const int64_t tilesA = (nA + kFlatA * kThreads - 1) / (kFlatA * kThreads);
    const int64_t tilesBC = (nB + nC + kThreads - 1) / kThreads;
    const int64_t n = nA + nB + nC;
    grid_launch_dependents();
    // records are plan tables, read before grid_dependency_wait(); forces after it
    // one tile per block, the grid covering every tile: without a grid-stride
    // loop the paths are straight-line and the kernel fits in 64 registers
    // (four resident blocks per SM; with the loop it needed 79, three blocks)
    const int64_t bb = blockIdx.x;
    if (bb >= tilesA + tilesBC) return;
    {
        if (bb >= tilesBC) {
            const int64_t m0 = (bb - tilesBC) * kFlatA * kThreads + threadIdx.x;
            if (ahead > 0 && bb + ahead < tilesA + tilesBC) {
                const int64_t n0 = (bb + ahead - tilesBC) * kFlatA * kThreads + threadIdx.x;
#pragma unroll
                for (int e = 0; e < kFlatA; e++)
                    if (n0 + e * kThreads < nA) prefetch_table(recA + n0 + e * kThreads);
            }
            int32_t home[kFlatA], ent[kFlatA][3];
            int kk[kFlatA];
#pragma unroll
            for (int e = 0; e < kFlatA; e++) {
                const int64_t m = m0 + e * kThreads;
                const int4 r = m < nA ? __ldg(recA + m) : make_int4(0, 0, 0, 0);
                home[e] = r.x & kNodeMask;
                ent[e][0] = r.y;
                ent[e][1] = r.z;
                ent[e][2] = r.w;
                const int k = (int)((unsigned)r.x >> kNodeBits);
                kk[e] = m < nA ? checked_copies<3>(home[e], k, ent[e], n_slots, err) : 0;
            }
            // first wave of a grid of more than one wave: this thread's force
            // lines into L2 while the kernel ahead drains (as in the
            // coordinate kernel).  The force kernel alone on the 1M-atom
            // system 10.2 -> 9.6 us, the 3M x + f 50.6 -> 49.8 us; a one-wave
            // grid (24k atoms) gains nothing, its prefetches only compete
            // with the kernel ahead.
            if (bb < ahead && tilesA + tilesBC > ahead) {
#pragma unroll
                for (int e = 0; e < kFlatA; e++) {
                    if (kk[e] > 0) prefetch_table(f + 3 * (int64_t)home[e]);
#pragma unroll
                    for (int j = 0; j < 3; j++)
                        if (j < kk[e]) prefetch_table(f + 3 * (int64_t)(ent[e][j] & kNodeMask));
                }
            }
            grid_dependency_wait();
            // the replacement block's trees: its records (prefetched above,
            // so L2 hits by now) give the force lines to prefetch, while this
            // thread's own loads are in flight.  Only for grids of at most two
            // waves: with more the blocks run bandwidth-bound and the extra
            // requests cost more than the latency they hide (1M-atom system
            // force kernel 10.95 -> 10.17 us; the 3M system 34.2 us with the
            // prefetch on every wave against 33.4 without).
            const int64_t nf = (bb + ahead - tilesBC) * kFlatA * kThreads + threadIdx.x;
            const bool fut = ahead > 0 && bb + ahead < tilesA + tilesBC && tilesA + tilesBC <= 2 * ahead;
            auto mid = [&]() {
                if (!fut) return;
#pragma unroll
                for (int e = 0; e < kFlatA; e++) {
                    const int64_t m = nf + e * kThreads;
                    if (m >= nA) continue;
                    const int4 r = __ldg(recA + m);
                    const int k = (int)((unsigned)r.x >> kNodeBits);
                    const int32_t node[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const int64_t slot = node[j] & kNodeMask;
                        if (j <= k && slot < n_slots) prefetch_table(f + 3 * slot);
                    }
                }
            };
            reduce_trees<3, kFlatA>(f, home, kk, ent, mid);
            return;
        }
        const int64_t m = nA + bb * kThreads + threadIdx.x;
        if (m >= n) return;  // touches nothing
        if (m < nA + nB) {
            const int4 r0 = __ldg(recB + 3 * (m - nA)), r1 = __ldg(recB + 3 * (m - nA) + 1);
            const int4 r2 = KB > 7 ? __ldg(recB + 3 * (m - nA) + 2) : make_int4(0, 0, 0, 0);
            const int32_t all[11] = {r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w, r2.x, r2.y, r2.z, r2.w};
            int32_t ent[KB];
#pragma unroll
            for (int j = 0; j < KB; j++) ent[j] = all[j];
            const int kb = checked_copies<KB>(r0.x & kNodeMask, (int)((unsigned)r0.x >> kNodeBits), ent,
                                              n_slots, err);
            grid_dependency_wait();
            reduce_tree<KB>(f, r0.x & kNodeMask, kb, ent);
        } else {
            const int4 r = __ldg(recC + (m - nA - nB));
            grid_dependency_wait();
            if constexpr (KW > 0) {
                if (((unsigned)r.x >> kNodeBits) <= (unsigned)KW) {
                    // plans with deeper trees (several pulses per dim): up to
                    // KW copies in registers
                    int k = (int)((unsigned)r.x >> kNodeBits);
                    if (k > 0 && !in_range((int64_t)r.y + k - 1, n_fent, err)) k = 0;
                    int32_t ent[KW];
#pragma unroll
                    for (int j = 0; j < KW; j++) ent[j] = j < k ? __ldg(fent + r.y + j) : 0;
                    const int kc = checked_copies<KW>(r.x & kNodeMask, k, ent, n_slots, err);
                    reduce_tree<KW>(f, r.x & kNodeMask, kc, ent);
                    return;
                }
            }
            // every slot of this tree belongs to this thread alone: plain
            // sequential read-modify-write in the same order, through L2
            float* fh = f + 3 * (int64_t)(r.x & kNodeMask);
            int k = (int)((unsigned)r.x >> kNodeBits);
            const int s0 = r.y;
            if (k > 0 && !(in_range(r.x & kNodeMask, n_slots, err) &&
                           in_range((int64_t)s0 + k - 1, n_fent, err)))
                k = 0;
            for (int j = 0; j < k; j++) {
                const int32_t e = __ldg(fent + s0 + j);
                const int par = (int)((unsigned)e >> kNodeBits);
                if (!in_range(e & kNodeMask, n_slots, err) || !in_range(par, k + 1, err)) continue;
                const float* fn = f + 3 * (int64_t)(e & kNodeMask);
                float* fp = par == 0 ? fh : f + 3 * (int64_t)(__ldg(fent + s0 + par - 1) & kNodeMask);
                const float n0 = __ldcg(fn), n1 = __ldcg(fn + 1), n2 = __ldcg(fn + 2);
                __stcg(fp, __ldcg(fp) + n0);
                __stcg(fp + 1, __ldcg(fp + 1) + n1);
                __stcg(fp + 2, __ldcg(fp + 2) + n2);
            }
        }
    }
}


int blocks_for(int64_t n, int num_sms) {
    return (int)std::max<int64_t>(1, std::min<int64_t>((n + kThreads - 1) / kThreads,
                                                       (int64_t)num_sms * 16));
}

}  // namespace

void free_flat(halo_plan* pl) {
    dev_free(pl->d_stage_buf);
    pl->cap_stage_buf = pl->n_stage_buf = 0;
    dev_free(pl->d_xflat);
    dev_free(pl->d_xflat_items);
    dev_free(pl->d_fown);
    dev_free(pl->d_fstart);
    dev_free(pl->d_fent);
    dev_free(pl->d_flat_pool32);
    dev_free(pl->d_flat_pool8);
    for (int c = 0; c < 3; c++) {
        dev_free(pl->d_frec[c]);
        pl->n_rec[c] = 0;
        pl->cap_frec[c] = 0;
    }
    pl->cap_xflat = pl->cap_xflat_items = pl->cap_fent = pl->cap_fown = pl->cap_fstart = 0;
    pl->cap_pool32 = pl->cap_pool8 = 0;
    pl->flat_ready = false;
    pl->n_xflat_items = 0;
    pl->n_owners = 0;
    pl->max_copies = 0;
}

namespace {
// Scratch of the FLAT table build, carved from two pools kept in the plan.
struct FlatScratch {
    int32_t *owner, *parent, *ncopies, *entry_pos, *rank, *tmp;
    int32_t* xbase;   // per domain: coordinate-table offset of halo slot 0, minus the slot
    int64_t* sums;    // int64 tile sums + grand total
    int32_t* misc;    // [0] largest copy list, [1] error
    int64_t* misc64;  // [0] copies | owners << 32, [1] class-A | class-B records << 32
    int8_t *hop, *code;
};

int flat_scratch(halo_plan* pl, FlatScratch* f) {
    const int64_t nl = pl->n_local_total, H = pl->n_halo_total;
    // int32 arrays start on 16-byte boundaries (the scans load and store them
    // 16 bytes at a time)
    const int64_t nl4 = (nl + 3) & ~(int64_t)3;
    const int64_t nsums = nl / kScanTile + 2;
    const int64_t off_xbase = 5 * nl4 + ((std::max<int64_t>(H, 1) + 1 + 3) & ~(int64_t)3);
    const int64_t off_sums = (off_xbase + pl->n_dom + 1) & ~(int64_t)1;  // 8-byte aligned
    HALO_TRY(dev_reserve(&pl->d_flat_pool32, &pl->cap_pool32, off_sums + 2 * nsums + 16));
    HALO_TRY(dev_reserve(&pl->d_flat_pool8, &pl->cap_pool8, 2 * nl));
    f->owner = pl->d_flat_pool32;
    f->parent = f->owner + nl4;
    f->ncopies = f->parent + nl4;
    f->entry_pos = f->ncopies + nl4;
    f->rank = f->entry_pos + nl4;
    f->tmp = f->rank + nl4;
    f->xbase = pl->d_flat_pool32 + off_xbase;
    f->sums = reinterpret_cast<int64_t*>(pl->d_flat_pool32 + off_sums);
    f->misc = pl->d_flat_pool32 + off_sums + 2 * nsums;
    f->misc64 = reinterpret_cast<int64_t*>(f->misc + 8);
    f->hop = pl->d_flat_pool8;
    f->code = f->hop + nl;
    return HALO_OK;
}
}  // namespace

int launch_flat_chains(halo_plan* pl, cudaStream_t st) {
    const int nd = pl->n_dom;
    if (pl->n_local_total >= ((int64_t)1 << kNodeBits)) return HALO_ECAPACITY;
    // coordinate items: halo range of every domain, in chunks of kXT * E
    // slots.  E = 2 unless that needs more than two waves of resident blocks,
    // then 3 (measured, x + f back to back, 128-thread blocks: the 1M-atom
    // system 18.4 us at E = 2 against 18.8, 19.4 and 18.8 at E = 3, 4 and 1,
    // where several small waves let the force kernel's blocks start early;
    // the 3M system 53.9 at E = 3 against 54.5 at E = 2).
    if (pl->occ_flat_x <= 0)
        HALO_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&pl->occ_flat_x, flat_x_kernel<2>, kXT, 0));
    int64_t items2 = 0;
    for (int D = 0; D < nd; D++)
        items2 += ((int64_t)pl->n_local[D] - pl->n_home[D] + 2 * kXT - 1) / (2 * kXT);
    const int E = items2 <= 2 * (int64_t)pl->num_sms * pl->occ_flat_x ? 2 : 3;
    pl->flat_x_e = E;
    const int kFlatChunk = kXT * E;
    // item b = {table offset b * kFlatChunk, first halo slot, count}: the
    // table is padded to whole chunks so a block can address its entries
    // from its index alone (the items are written on the device)
    int64_t n_items = 0;
    for (int D = 0; D < nd; D++)
        n_items += ((int64_t)pl->n_local[D] - pl->n_home[D] + kFlatChunk - 1) / kFlatChunk;
    pl->n_xflat_items = (int)n_items;
    HALO_TRY(dev_reserve(&pl->d_xflat_items, &pl->cap_xflat_items, n_items));
    HALO_TRY(dev_reserve(&pl->d_xflat, &pl->cap_xflat, std::max<int64_t>(n_items * kFlatChunk, 1)));
    FlatScratch f;
    HALO_TRY(flat_scratch(pl, &f));
    HALO_CUDA(cudaMemsetAsync(f.ncopies, 0, sizeof(int32_t) * pl->n_local_total, st));
    HALO_CUDA(cudaMemsetAsync(f.misc, 0, sizeof(int32_t) * 16, st));
    if (n_items > 0)
        HALO_CUDA(launch_dependent_shm(xflat_items_kernel, dim3((unsigned)((nd + 31) / 32)), dim3(1024), 0, st,
                                       domain_tables(pl), nd, pl->P, kFlatChunk, pl->d_xflat_items, f.xbase));
    for (int p = 0; p < pl->P; p++) {
        const unsigned gx = (unsigned)std::min(std::max(pl->max_chunks[p], 1), 1024);
        HALO_CUDA(launch_dependent_shm(chain_pulse_kernel, dim3(gx, nd), dim3(kThreads), 0, st,
                                       (const SPDesc*)pl->d_sp, (const int32_t*)pl->d_maps, f.owner,
                                       f.parent, f.hop, f.code, (const int32_t*)f.xbase, pl->d_xflat,
                                       f.ncopies, f.rank, pl->P, p, (int)pl->pulse_dim[p]));
    }
    HALO_CUDA(cudaGetLastError());
    pl->flat_chains_ready = true;
    return HALO_OK;
}

int prepare_flat(halo_plan* pl, cudaStream_t st) {
    pl->flat_ready = false;  // buffers are kept (grow-only) across rebuilds
    const int64_t nl = pl->n_local_total, H = pl->n_halo_total;
    if (nl >= ((int64_t)1 << kNodeBits)) return HALO_ECAPACITY;
    // the coordinate items, the forwarding chains and the coordinate table
    // need only the pulse descriptors and the sizes: a rebuild launches them
    // as soon as those are known (before the host's own copy of the plan is
    // built), else they are launched here
    if (!pl->flat_chains_ready) HALO_TRY(launch_flat_chains(pl, st));
    pl->flat_chains_ready = false;
    const int64_t n_items = pl->n_xflat_items;
    HALO_TRY(dev_reserve(&pl->d_fent, &pl->cap_fent, H));
    // owner tables sized by bounds (every halo slot is one copy of one owner:
    // at most H owners, H / 4 with 4..11 copies, H / 12 with more), so that
    // no count has to come back to the host before the end
    HALO_TRY(dev_reserve(&pl->d_fown, &pl->cap_fown, H));
    HALO_TRY(dev_reserve(&pl->d_fstart, &pl->cap_fstart, H + 1));
    HALO_TRY(dev_reserve(&pl->d_frec[0], &pl->cap_frec[0], H));
    HALO_TRY(dev_reserve(&pl->d_frec[1], &pl->cap_frec[1], 3 * (H / 4 + 1)));
    HALO_TRY(dev_reserve(&pl->d_frec[2], &pl->cap_frec[2], H / 12 + 1));

    FlatScratch f;
    HALO_TRY(flat_scratch(pl, &f));
    int32_t* owner = f.owner;
    int32_t* parent = f.parent;
    int32_t* ncopies = f.ncopies;
    int32_t* entry_pos = f.entry_pos;
    int32_t* rank = f.rank;
    int32_t* tmp = f.tmp;
    int64_t* sums = f.sums;
    int32_t* misc = f.misc;
    int64_t* misc64 = f.misc64;
    int8_t* hop = f.hop;

    // pinned staging: words read back at the end
    int64_t* hw = nullptr;
    {
        void* hs = nullptr;
        HALO_TRY(host_stage(pl, 256, &hs));
        hw = static_cast<int64_t*>(hs);  // 8 words
    }
    int rc = HALO_OK;
    do {
        const int gh = blocks_for(std::max<int64_t>(H, 1), pl->num_sms);
        // entry offsets of every slot's copy list and, from the same scan,
        // the owner list (fown, fstart); the grand total (copies, owners)
        // stays on the device
        if ((rc = pair_scan<0>(ncopies, nl, nullptr, sums, entry_pos, nullptr, misc64, st, pl->d_fown,
                               pl->d_fstart)) != HALO_OK)
            break;
        if (n_items > 0)
            if ((rc = cuda_code(launch_dependent_shm(
                     owner_fill_kernel, dim3((unsigned)std::min<int64_t>(n_items, 8 * (int64_t)pl->num_sms)),
                     dim3(kThreads), 0, st, (const int4*)pl->d_xflat_items, (int)n_items,
                     (const int32_t*)owner, (const int32_t*)entry_pos, (const int32_t*)rank, tmp))) != HALO_OK)
                break;
        // record classes (A: <= 3 copies, B: 4..11, C: more): positions in
        // each class from one paired scan of the owners' copy counts, then the
        // sort writes every owner's record there
        int32_t* posA = entry_pos;  // scratch reuse: owner_fill has read entry_pos
        int32_t* posB = ncopies;    // and the copy-count scan ncopies
        if ((rc = pair_scan<1>(pl->d_fstart, std::max<int64_t>(H, 1), misc64, sums, posA, posB,
                               misc64 + 1, st)) != HALO_OK)
            break;
        // class A here; classes B and C (listed in the ranks' place: owner_fill
        // has read them) in a second pass
        int32_t* listB = rank;
        int32_t* listC = rank + (H / 4 + 1);
        if ((rc = cuda_code(launch_dependent_shm(
                 owner_sort_kernel, dim3(gh), dim3(kThreads), 0, st, (const int32_t*)pl->d_fown,
                 (const int32_t*)pl->d_fstart, (const int32_t*)tmp, (const int32_t*)parent,
                 (const int8_t*)hop, (const int64_t*)misc64, (const int32_t*)posA, (const int32_t*)posB,
                 pl->d_frec[0], listB, listC, misc, misc + 1))) != HALO_OK)
            break;
        // the summary words come back through the mapped staging (written by
        // the last sort block), else with a copy
        int32_t* host_out = static_cast<int32_t*>(pl->h_stage_dev);
        if ((rc = cuda_code(launch_dependent_shm(
                 owner_sort_bc_kernel, dim3(blocks_for(H / 4 + 1, pl->num_sms)), dim3(kThreads), 0, st,
                 (const int32_t*)pl->d_fown, (const int32_t*)pl->d_fstart, (const int32_t*)tmp,
                 (const int32_t*)parent, (const int8_t*)hop, (const int64_t*)misc64,
                 (const int32_t*)posA, (const int32_t*)posB, (const int32_t*)listB,
                 (const int32_t*)listC, pl->d_frec[1], pl->d_frec[2], pl->d_fent, misc + 1, misc,
                 host_out))) != HALO_OK)
            break;
        // the one synchronisation: counts, largest list, error
        if (!host_out &&
            (rc = cuda_code(cudaMemcpyAsync(hw, misc, 8 * sizeof(int32_t) + 2 * sizeof(int64_t),
                                            cudaMemcpyDeviceToHost, st))) != HALO_OK)
            break;
        if ((rc = cuda_code(cudaStreamSynchronize(st))) != HALO_OK) break;
        if ((rc = cuda_code(cudaGetLastError())) != HALO_OK) break;
        const int32_t* info = reinterpret_cast<const int32_t*>(hw);
        const int64_t tot_copies = hw[4] & 0xffffffffll, n_owners = hw[4] >> 32;
        if (info[1] != 0 || tot_copies != H) {  // every halo slot is one copy of one owner
            rc = HALO_ECAPACITY;
            break;
        }
        pl->n_owners = n_owners;
        pl->max_copies = info[0];
        pl->n_rec[0] = hw[5] & 0xffffffffll;
        pl->n_rec[1] = hw[5] >> 32;
        pl->n_rec[2] = n_owners - pl->n_rec[0] - pl->n_rec[1];
    } while (false);
    if (rc != HALO_OK) return rc;
    pl->flat_ready = true;
    return HALO_OK;
}

int launch_stepwise_x(halo_plan* pl, float* xyz, cudaStream_t st) {
    for (int p = 0; p < pl->P; p++) {
        const unsigned gx = (unsigned)std::min(std::max(pl->max_chunks[p], 1), 1024);
        const cudaError_t e = launch_dependent(step_x_kernel, dim3(gx, pl->n_dom), dim3(kThreads), st,
                                               (const SPDesc*)pl->d_sp, (const int32_t*)pl->d_maps, xyz,
                                               pl->P, p, pl->n_local_total, pl->d_err);
        if (e != cudaSuccess) return cuda_code(e);
        pl->launches_x++;
    }
    return cuda_code(cudaGetLastError());
}

int launch_stepwise_f(halo_plan* pl, float* f, cudaStream_t st) {
    for (int p = pl->P - 1; p >= 0; p--) {
        const unsigned gx = (unsigned)std::min(std::max(pl->max_chunks[p], 1), 1024);
        const cudaError_t e = launch_dependent(step_f_kernel, dim3(gx, pl->n_dom), dim3(kThreads), st,
                                               (const SPDesc*)pl->d_sp, (const int32_t*)pl->d_maps, f,
                                               pl->P, p, pl->n_local_total, pl->d_err);
        if (e != cudaSuccess) return cuda_code(e);
        pl->launches_f++;
    }
    return cuda_code(cudaGetLastError());
}

int prepare_staged(halo_plan* pl) {
    int64_t n = 0;
    for (const SPDesc& d : pl->sp) n = std::max<int64_t>(n, d.map_off + d.send);
    pl->n_stage_buf = n;
    return dev_reserve(&pl->d_stage_buf, &pl->cap_stage_buf, std::max<int64_t>(3 * n, 1));
}

int launch_staged_x(halo_plan* pl, float* xyz, cudaStream_t st) {
    if (!pl->d_stage_buf) return HALO_EINVAL;
    for (int p = 0; p < pl->P; p++) {
        const unsigned gx = (unsigned)std::min(std::max(pl->max_chunks[p], 1), 1024);
        staged_pack_x_kernel<<<dim3(gx, pl->n_dom), kThreads, 0, st>>>(
            pl->d_sp, pl->d_maps, xyz, pl->d_stage_buf, pl->P, p, pl->n_local_total, pl->n_stage_buf,
            pl->d_err);
        pl->launches_x++;
        HALO_CUDA(cudaStreamSynchronize(st));  // the host waits for the send buffer
        staged_move_kernel<true><<<dim3(std::min(3 * gx, 1024u), pl->n_dom), kThreads, 0, st>>>(
            pl->d_sp, xyz, pl->d_stage_buf, pl->P, p, pl->n_local_total, pl->n_stage_buf, pl->d_err);
        pl->launches_x++;
        HALO_CUDA(cudaStreamSynchronize(st));  // and for the message before the next pulse
    }
    return cuda_code(cudaGetLastError());
}

int launch_staged_f(halo_plan* pl, float* f, cudaStream_t st) {
    if (!pl->d_stage_buf) return HALO_EINVAL;
    for (int p = pl->P - 1; p >= 0; p--) {
        const unsigned gx = (unsigned)std::min(std::max(pl->max_chunks[p], 1), 1024);
        staged_move_kernel<false><<<dim3(std::min(3 * gx, 1024u), pl->n_dom), kThreads, 0, st>>>(
            pl->d_sp, f, pl->d_stage_buf, pl->P, p, pl->n_local_total, pl->n_stage_buf, pl->d_err);
        pl->launches_f++;
        HALO_CUDA(cudaStreamSynchronize(st));  // the message has arrived
        staged_unpack_f_kernel<<<dim3(gx, pl->n_dom), kThreads, 0, st>>>(
            pl->d_sp, pl->d_maps, f, pl->d_stage_buf, pl->P, p, pl->n_local_total, pl->n_stage_buf,
            pl->d_err);
        pl->launches_f++;
        HALO_CUDA(cudaStreamSynchronize(st));  // unpacked before the next pulse's send
    }
    return cuda_code(cudaGetLastError());
}

int launch_flat_x(halo_plan* pl, float* xyz, cudaStream_t st) {
    if (pl->n_xflat_items == 0) return HALO_OK;
    auto* k = pl->flat_x_e == 3 ? flat_x_kernel<3> : flat_x_kernel<2>;
    if (pl->ahead_x[pl->flat_x_e] == 0) {
        int occ = 0;
        HALO_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kXT, 0));
        pl->ahead_x[pl->flat_x_e] = std::max(occ, 1) * pl->num_sms;
    }
    const cudaError_t e = launch_dependent(k, dim3(pl->n_xflat_items), dim3(kXT), st, xyz,
                                           (const int32_t*)pl->d_xflat, (const int4*)pl->d_xflat_items,
                                           pl->box[0], pl->box[1], pl->box[2], pl->n_local_total,
                                           pl->d_err, pl->ahead_x[pl->flat_x_e]);
    if (e != cudaSuccess) return cuda_code(e);
    pl->launches_x++;
    return HALO_OK;
}

int launch_flat_f(halo_plan* pl, float* f, cudaStream_t st) {
    if (pl->n_owners == 0) return HALO_OK;
    // class A goes kFlatA owners per thread, classes B and C one per thread
    const int64_t tilesA = (pl->n_rec[0] + kFlatA * kThreads - 1) / (kFlatA * kThreads);
    const int64_t tilesBC = (pl->n_rec[1] + pl->n_rec[2] + kThreads - 1) / kThreads;
    const int gb = (int)std::max<int64_t>(1, tilesA + tilesBC);
    const int ki = pl->max_copies <= 7 ? 0 : pl->max_copies <= 11 ? 1 : 2;
    auto* k = ki == 0 ? flat_f_kernel<7, 0> : ki == 1 ? flat_f_kernel<11, 0> : flat_f_kernel<11, 16>;
    if (pl->ahead_f[ki] == 0) {
        int occ = 0;
        HALO_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kThreads, 0));
        pl->ahead_f[ki] = std::max(occ, 1) * pl->num_sms;
    }
    const cudaError_t e = launch_dependent(k, dim3(gb), dim3(kThreads), st, f, (const int4*)pl->d_frec[0],
                                           pl->n_rec[0], (const int4*)pl->d_frec[1], pl->n_rec[1],
                                           (const int4*)pl->d_frec[2], pl->n_rec[2],
                                           (const int32_t*)pl->d_fent, pl->n_local_total,
                                           pl->n_halo_total, pl->d_err, (int64_t)pl->ahead_f[ki]);
    if (e != cudaSuccess) return cuda_code(e);
    pl->launches_f++;
    return HALO_OK;
}

}  // namespace halo
