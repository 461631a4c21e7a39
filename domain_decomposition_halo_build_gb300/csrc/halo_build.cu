// halo_build.cu -- device-side construction of the per-pulse index maps.
//
// Page "Redesigning GROMACS Halo Exchange: Improving Strong Scaling with
// GPU-initiated NVSHMEM" (review), section 3 and Algorithm 1: every domain owns
// its home atoms; for each pulse, the atoms of a sender domain that lie within
// the cut-off of its lower face are listed in an index map (PulseData.indexMap,
// sendSize), which the receiver appends to its halo at atomOffset, shifted by
// coordShift across the periodic boundary.  Forwarding (eighth shell): pulse 0
// of a dim selects among home atoms plus all halo received in earlier dims,
// pulse k >= 1 only among the slots received in pulse k-1 of the same dim.
// Algorithm 4: depOffset splits each map into entries that are home atoms
// (independent) and entries that arrived in earlier pulses (dependent).
//
// Device pipeline (one stream, one host synchronisation at the end):
//   1. home partition: a histogram of domain ids per block tile (per-warp
//      shared histograms), exclusive scan, stable scatter (each tile ranked in
//      shared memory: warp match + running per-domain counters) -> every
//      domain's home atoms in input order, in a home-compact region;
//   2. per pulse: count kernel (predicate per candidate, with the optional
//      corner test; its last block scans the unit counts into offsets, sizes
//      and receiver offsets), write kernel (stable warp ballot compaction -> ascending index map +
//      the new halo coordinates);
//   3. finalize: dense bases, pulse descriptors; the metadata back to the
//      host.
// Index maps hold domain-relative local indices, so the dense relayout touches
// none of them.
#include <math.h>
#include <string.h>

#include <algorithm>

#include "halo_device.cuh"
#include "halo_internal.cuh"

namespace halo {
namespace {

// ---- packed metadata (int64 entries) -----------------------------------------
struct Meta {
    int64_t* flags;     // [0] capacity overflow, [1] bad domain id
    int64_t* n_home;    // n_dom
    int64_t* hstart;    // n_dom: first home-compact slot of each domain
    int64_t* base;      // n_dom: first dense slot of each domain
    int64_t* own_off;   // n_dom*(P+1): first local index of each received slice; [P] = n_local
    int64_t* recv_pos;  // n_dom*P: build-buffer slot of each received slice
    int64_t* send;      // n_dom*P
    int64_t* split;     // n_dom*P
    int64_t* map_pos;   // n_dom*P: build-buffer slot of the sender's output
    int64_t* region;    // P+1: first build-buffer slot of each pulse's output region
};

size_t meta_count(int nd, int P) {
    return 4 + 3 * (size_t)nd + (size_t)nd * (P + 1) + 4 * (size_t)nd * P + (P + 1);
}

Meta meta_ptrs(void* m, int nd, int P) {
    int64_t* q = (int64_t*)m;
    Meta r;
    r.flags = q;
    q += 4;
    r.n_home = q;
    q += nd;
    r.hstart = q;
    q += nd;
    r.base = q;
    q += nd;
    r.own_off = q;
    q += (size_t)nd * (P + 1);
    r.recv_pos = q;
    q += (size_t)nd * P;
    r.send = q;
    q += (size_t)nd * P;
    r.split = q;
    q += (size_t)nd * P;
    r.map_pos = q;
    q += (size_t)nd * P;
    r.region = q;
    return r;
}


__device__ __forceinline__ int cell_of(int D, int d, int nx, int ny) {
    return d == 0 ? D % nx : (d == 1 ? (D / nx) % ny : D / (nx * ny));
}


// The lanes of the warp whose domain id equals this lane's (valid lanes only;
// an invalid lane's result is not used): one ballot per bit of the id, so
// the cost is fixed (nbits + 1 ballots) where the match instruction's grows
// with the number of distinct ids among the 32 lanes.
__device__ __forceinline__ unsigned same_domain_lanes(int d, bool valid, int nbits) {
    unsigned m = __ballot_sync(kFull, valid);
    for (int b = 0; b < nbits; b++) {
        const bool bit = ((d >> b) & 1) != 0;
        const unsigned bb = __ballot_sync(kFull, bit);
        m &= bit ? bb : ~bb;
    }
    return m;
}

// ---- 1. home partition ------------------------------------------------------------
// A block of W warps covers the block tile b of W * wtile atoms; warp w its
// sub-tile [(b*W + w)*wtile, ... + wtile) (wtile a multiple of 128).  Each
// warp counts its sub-tile into its own shared histogram (shared-memory
// atomics); the block writes one count per domain: tile-major,
// counts[b*nd + D] (tiled scatter), or domain-major, counts[D*nbt + b], so
// that one exclusive scan gives every (domain, block tile) start, and then,
// if wcounts is given, every warp's counts, wcounts[(b*W + w)*nd + D]
// (contiguous per block, for the direct scatter).
__global__ void home_hist_kernel(const int32_t* __restrict__ dom, int64_t n, int nd, int64_t nbt,
                                 int wtile, int tile_major, int32_t* __restrict__ counts,
                                 int32_t* __restrict__ wcounts, int64_t* __restrict__ flags) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    extern __shared__ int32_t sh[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int W = blockDim.x >> 5;
    int32_t* h = sh + (size_t)warp * nd;
    for (int i = lane; i < nd; i += 32) h[i] = 0;
    __syncwarp();
    const int64_t a0 = ((int64_t)blockIdx.x * W + warp) * wtile;
    bool bad = false;
    // four coalesced loads in flight per lane, then their counts
    constexpr int U = 4;
    for (int it = 0; it < wtile / 32; it += U) {
        int d[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t a = a0 + (it + u) * 32 + lane;
            d[u] = a < n ? __ldg(dom + a) : 0;
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            if (a0 + (it + u) * 32 + lane >= n) continue;
            if (d[u] < 0 || d[u] >= nd)
                bad = true;
            else
                atomicAdd(&h[d[u]], 1);
        }
    }
    if (bad) flags[1] = 1;
    __syncthreads();
    if (wcounts) {
        int32_t* wc = wcounts + (int64_t)blockIdx.x * W * nd;
        for (int i = threadIdx.x; i < W * nd; i += blockDim.x) wc[i] = sh[i];
    }
    for (int d = threadIdx.x; d < nd; d += blockDim.x) {
        int32_t t = 0;
        for (int w = 0; w < W; w++) t += sh[(size_t)w * nd + d];
        counts[tile_major ? (int64_t)blockIdx.x * nd + d : (int64_t)d * nbt + blockIdx.x] = t;
    }
}

// Stable scatter: every warp's start per domain is its block tile's start
// plus the counts of the warps before it; then each warp visits its atoms in
// input order, and within 32 atoms the rank among equal domain ids comes from
// the lanes with the same id (same_domain_lanes).
__global__ void home_scatter_kernel(const float* __restrict__ xyz, const int32_t* __restrict__ dom,
                                    int64_t n, int nd, int64_t nbt,
                                    const int32_t* __restrict__ offs,
                                    const int32_t* __restrict__ wcounts,
                                    int32_t* __restrict__ home_gid, float4* __restrict__ bxyz) {
    const int nbits = 32 - __clz(max(nd - 1, 0));  // bits of a domain id
    extern __shared__ int32_t sh[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int W = blockDim.x >> 5;
    int32_t* run = sh + (size_t)warp * nd;
    const int32_t* wc = wcounts + (int64_t)blockIdx.x * W * nd;
    for (int d = threadIdx.x; d < nd; d += blockDim.x) {
        int32_t acc = offs[(int64_t)d * nbt + blockIdx.x];
        for (int w = 0; w < W; w++) {
            sh[(size_t)w * nd + d] = acc;
            acc += wc[(size_t)w * nd + d];
        }
    }
    __syncthreads();
    const int64_t a0 = ((int64_t)blockIdx.x * W + warp) * kHistTile;
    const unsigned lt = lanemask_lt();
    // four rounds of 32 atoms per step: their ids and coordinates are loaded
    // first (independent loads in flight), then the rounds are placed in
    // order, so the partition stays stable
    constexpr int U = 4;
    for (int it = 0; it < kHistTile / 32; it += U) {
        int d[U];
        float c[U][3];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t a = a0 + (it + u) * 32 + lane;
            d[u] = -1;
            c[u][0] = c[u][1] = c[u][2] = 0.0f;
            if (a < n) {
                d[u] = __ldg(dom + a);
                if (d[u] < 0 || d[u] >= nd) d[u] = -1;
                c[u][0] = __ldg(xyz + 3 * a + 0);
                c[u][1] = __ldg(xyz + 3 * a + 1);
                c[u][2] = __ldg(xyz + 3 * a + 2);
            }
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t a = a0 + (it + u) * 32 + lane;
            const unsigned peers = same_domain_lanes(d[u], d[u] >= 0, nbits);
            if (d[u] >= 0) {
                const int64_t pos = (int64_t)run[d[u]] + __popc(peers & lt);
                home_gid[pos] = (int32_t)a;
                // one 16-byte store: the coordinates, and no forwarding dims
                bxyz[pos] = make_float4(c[u][0], c[u][1], c[u][2], __int_as_float(0));
            }
            __syncwarp();
            if (d[u] >= 0 && lane == __ffs(peers) - 1) run[d[u]] += __popc(peers);
            __syncwarp();
        }
    }
}

// The stable scatter with the block's whole tile in shared memory.  Block b
// copies its T atoms' coordinates and domain ids into shared memory (16-byte
// asynchronous copies where the tile is 16-byte aligned, so every copy is in
// flight at once), counts them per warp sub-tile, ranks them (per-domain tile
// starts, then each warp's atoms in input order, 32 at a time, ranks among
// equal ids from same_domain_lanes) and writes every domain's run of the
// tile contiguously, from hstart[D] + pre[b*nd + D] (the column prefixes of
// the tile-major counts).  Several blocks fit on an SM, so one block's copies
// overlap another's ranking.
__host__ __device__ inline size_t tile_scatter_head(int W, int nd) {
    return ((((size_t)W * nd + 2 * (size_t)nd + 1) * sizeof(int32_t)) + 15) & ~(size_t)15;
}
__host__ __device__ inline size_t tile_scatter_smem(int W, int nd, int T) {
    // raw coordinates, raw domain ids, sorted position -> tile index
    return tile_scatter_head(W, nd) + (size_t)T * (3 * sizeof(float) + sizeof(int32_t) + sizeof(int16_t));
}

// Column prefixes of the tile-major counts: for domain d (a lane of a strip
// of 32 domains) and tile b, pre[b*nd + d] = the count of d's atoms in tiles
// before b; the warps of a block split the tiles into 32 contiguous ranges.
// Column totals are the home counts n_home[d].  The last block to finish
// (an atomic ticket in flags[2], zeroed with the metadata) scans them: every
// domain's first home slot hstart[d], own_off[d][0] = n_home[d], region[0].
__global__ void __launch_bounds__(1024) home_colscan_kernel(const int32_t* __restrict__ counts,
                                                            int64_t nbt, int nd, int P, int64_t n,
                                                            int32_t* __restrict__ pre, Meta m) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    __shared__ int32_t part[32][33];
    __shared__ int last;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int d = blockIdx.x * 32 + lane;
    const int64_t b0 = nbt * w / 32, b1 = nbt * (w + 1) / 32;
    int32_t s = 0;
    if (d < nd) {
        int64_t b = b0;
        for (; b + 4 <= b1; b += 4) {
            const int32_t c0 = counts[b * nd + d], c1 = counts[(b + 1) * nd + d];
            const int32_t c2 = counts[(b + 2) * nd + d], c3 = counts[(b + 3) * nd + d];
            s += (c0 + c1) + (c2 + c3);
        }
        for (; b < b1; b++) s += counts[b * nd + d];
    }
    part[w][lane] = s;
    __syncthreads();
    int32_t acc = 0, tot = 0;
    for (int q = 0; q < 32; q++) {
        const int32_t v = part[q][lane];
        acc += q < w ? v : 0;
        tot += v;
    }
    if (d < nd) {
        int64_t b = b0;
        for (; b + 4 <= b1; b += 4) {  // four loads in flight, then their prefixes
            const int32_t c0 = counts[b * nd + d], c1 = counts[(b + 1) * nd + d];
            const int32_t c2 = counts[(b + 2) * nd + d], c3 = counts[(b + 3) * nd + d];
            pre[b * nd + d] = acc;
            pre[(b + 1) * nd + d] = acc + c0;
            pre[(b + 2) * nd + d] = acc + c0 + c1;
            pre[(b + 3) * nd + d] = acc + c0 + c1 + c2;
            acc += (c0 + c1) + (c2 + c3);
        }
        for (; b < b1; b++) {
            pre[b * nd + d] = acc;
            acc += counts[b * nd + d];
        }
        if (w == 0) m.n_home[d] = tot;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0)
        last = atomicAdd(reinterpret_cast<unsigned long long*>(m.flags + 2), 1ull) == gridDim.x - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
    int64_t carry = 0;
    for (int D0 = 0; D0 < nd; D0 += 1024) {
        const int D = D0 + threadIdx.x;
        const int64_t v = D < nd ? __ldcg(m.n_home + D) : 0;
        int64_t t;
        const int64_t p0 = block_exclusive_scan<1024>(v, &t);
        if (D < nd) {
            m.hstart[D] = carry + p0;
            m.own_off[(int64_t)D * (P + 1)] = v;
        }
        carry += t;
    }
    if (threadIdx.x == 0) m.region[0] = n;
}

constexpr int kScatterThreads = 512;  // threads (16 warp sub-tiles) per tiled scatter block

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}

__global__ void __launch_bounds__(kScatterThreads) home_scatter_tile_kernel(
    const float* __restrict__ xyz, const int32_t* __restrict__ dom, int64_t n, int nd, int T,
    int vec, const int32_t* __restrict__ pre, const int64_t* __restrict__ hstart,
    int32_t* __restrict__ home_gid, float4* __restrict__ bxyz) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    const int nbits = 32 - __clz(max(nd - 1, 0));  // bits of a domain id
    extern __shared__ __align__(16) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int W = kScatterThreads / 32;
    int32_t* whist = reinterpret_cast<int32_t*>(smem);  // W * nd: per warp and domain
    int32_t* lstart = whist + (size_t)W * nd;           // nd + 1: tile start of each domain
    int32_t* gstart = lstart + nd + 1;                  // nd: the domain run's first home slot
    float* rx = reinterpret_cast<float*>(smem + tile_scatter_head(W, nd));
    int32_t* rd = reinterpret_cast<int32_t*>(rx + 3 * (size_t)T);
    int16_t* perm = reinterpret_cast<int16_t*>(rd + T);
    const int64_t a0 = (int64_t)blockIdx.x * T;
    const int cnt = (int)min((int64_t)T, n - a0);
    const float* gx = xyz + 3 * a0;
    const int32_t* gd = dom + a0;
    // 1. the raw tile into shared memory
    const int nf = 3 * cnt;
    int vf = 0, vd = 0;
    if (vec) {
        vf = nf >> 2;
        vd = cnt >> 2;
        for (int i = threadIdx.x; i < vf; i += kScatterThreads) cp_async16(rx + 4 * i, gx + 4 * i);
        for (int i = threadIdx.x; i < vd; i += kScatterThreads) cp_async16(rd + 4 * i, gd + 4 * i);
    }
    for (int i = 4 * vf + threadIdx.x; i < nf; i += kScatterThreads) rx[i] = __ldg(gx + i);
    for (int i = 4 * vd + threadIdx.x; i < cnt; i += kScatterThreads) rd[i] = __ldg(gd + i);
    for (int d = threadIdx.x; d < nd; d += kScatterThreads)
        gstart[d] = (int32_t)hstart[d] + pre[(int64_t)blockIdx.x * nd + d];
    for (int i = threadIdx.x; i < W * nd; i += kScatterThreads) whist[i] = 0;
    if (vec) asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
    // 2. per-warp counts of the warp's sub-tile
    const int S = T / W;
    const int i0 = warp * S;
    for (int i = i0 + lane; i < i0 + S; i += 32) {
        if (i >= cnt) break;
        const int d = rd[i];
        if (d >= 0 && d < nd) atomicAdd(&whist[(size_t)warp * nd + d], 1);
    }
    __syncthreads();
    // 3. tile count per domain; each warp's start within its domain's run
    for (int d = threadIdx.x; d < nd; d += kScatterThreads) {
        int32_t acc = 0;
        for (int w = 0; w < W; w++) {
            const int32_t c = whist[(size_t)w * nd + d];
            whist[(size_t)w * nd + d] = acc;
            acc += c;
        }
        lstart[d] = acc;
    }
    __syncthreads();
    {
        // exclusive scan of the tile counts over the domains, two per thread
        // (the tiled path has nd <= 2 * kScatterThreads)
        const int d0 = 2 * threadIdx.x;
        const int32_t v0 = d0 < nd ? lstart[d0] : 0, v1 = d0 + 1 < nd ? lstart[d0 + 1] : 0;
        int64_t tot;
        const int64_t pre = block_exclusive_scan<kScatterThreads>(v0 + v1, &tot);
        if (d0 < nd) lstart[d0] = (int32_t)pre;
        if (d0 + 1 < nd) lstart[d0 + 1] = (int32_t)(pre + v0);
        if (threadIdx.x == 0) lstart[nd] = (int32_t)tot;
    }
    __syncthreads();
    for (int d = threadIdx.x; d < nd; d += kScatterThreads) {
        const int32_t l = lstart[d];
        for (int w = 0; w < W; w++) whist[(size_t)w * nd + d] += l;
    }
    __syncthreads();
    // 4. rank: each warp places its atoms in input order
    const unsigned lt = lanemask_lt();
    int32_t* run = whist + (size_t)warp * nd;
    for (int r = 0; r < S; r += 32) {
        const int i = i0 + r + lane;
        int d = i < cnt ? rd[i] : -1;
        if (d >= nd) d = -1;
        const unsigned peers = same_domain_lanes(d, d >= 0, nbits);
        if (d >= 0) perm[run[d] + __popc(peers & lt)] = (int16_t)i;
        __syncwarp();
        if (d >= 0 && lane == __ffs(peers) - 1) run[d] += __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    // 5. every domain's run of the tile, contiguous in the home-compact region
    const int total = lstart[nd];
    for (int j = threadIdx.x; j < total; j += kScatterThreads) {
        const int i = perm[j];
        const int d = rd[i];
        const int64_t g = (int64_t)gstart[d] + (j - lstart[d]);
        bxyz[g] = make_float4(rx[3 * i], rx[3 * i + 1], rx[3 * i + 2], __int_as_float(0));
        home_gid[g] = (int32_t)(a0 + i);
    }
}

// ---- generic int32 exclusive scan (three launches) ---------------------------------
__global__ void scan_reduce_kernel(const int32_t* __restrict__ in, int64_t n,
                                   int32_t* __restrict__ sums) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    const int64_t b0 = (int64_t)blockIdx.x * kScanTile;
    int64_t s = 0;
    for (int j = threadIdx.x; j < kScanTile; j += kThreads) {
        const int64_t i = b0 + j;
        if (i < n) s += in[i];
    }
    int64_t tot;
    block_exclusive_scan<kThreads>(s, &tot);
    if (threadIdx.x == 0) sums[blockIdx.x] = (int32_t)tot;
}

__global__ void scan_top_kernel(int32_t* __restrict__ sums, int64_t nb) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    int64_t carry = 0;
    for (int64_t b = 0; b < nb; b += 1024) {
        const int64_t i = b + threadIdx.x;
        const int64_t v = i < nb ? sums[i] : 0;
        int64_t tot;
        const int64_t pre = block_exclusive_scan<1024>(v, &tot);
        if (i < nb) sums[i] = (int32_t)(carry + pre);
        carry += tot;
    }
}

__global__ void __launch_bounds__(kThreads) scan_down_kernel(const int32_t* __restrict__ in,
                                                             int32_t* __restrict__ out, int64_t n,
                                                             const int32_t* __restrict__ sums) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    // each warp walks a contiguous run of the tile 32 elements at a time
    // (coalesced), a shuffle scan per 32, warp totals scanned across the block
    constexpr int kWarps = kThreads / 32;
    constexpr int R = kScanTile / kThreads;
    __shared__ int64_t wsum[kWarps];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t r0 = (int64_t)blockIdx.x * kScanTile + (int64_t)w * 32 * R;
    int32_t v[R];
    int64_t s = 0;
#pragma unroll
    for (int r = 0; r < R; r++) {
        const int64_t i = r0 + r * 32 + lane;
        v[r] = i < n ? in[i] : 0;
        s += v[r];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
    if (lane == 0) wsum[w] = s;
    __syncthreads();
    int64_t carry = sums[blockIdx.x];
    for (int q = 0; q < w; q++) carry += wsum[q];
#pragma unroll
    for (int r = 0; r < R; r++) {
        int64_t x = v[r];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t y = __shfl_up_sync(kFull, x, o);
            if (lane >= o) x += y;
        }
        const int64_t i = r0 + r * 32 + lane;
        if (i < n) out[i] = (int32_t)(carry + x - v[r]);
        carry += __shfl_sync(kFull, x, 31);
    }
}

// Per-domain home counts and starts from the scanned tile offsets; pulse state init.
__global__ void home_meta_kernel(const int32_t* __restrict__ offs, int64_t ntiles, int64_t n,
                                 int nd, int P, Meta m) {
    for (int D = blockIdx.x * blockDim.x + threadIdx.x; D < nd; D += gridDim.x * blockDim.x) {
        const int64_t h0 = offs[(int64_t)D * ntiles];
        const int64_t h1 = (D + 1 < nd) ? offs[(int64_t)(D + 1) * ntiles] : n;
        m.hstart[D] = h0;
        m.n_home[D] = h1 - h0;
        m.own_off[(int64_t)D * (P + 1)] = h1 - h0;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        m.region[0] = n;
        m.flags[0] = 0;
    }
}

// ---- 2. one pulse ---------------------------------------------------------------
struct PulseArgs {
    float4* bxyz;       // per build slot: x, y, z and (as int bits) the dims it was received across
    int32_t* maps;  // maps[slot - N]
    int64_t N;
    int64_t cap;    // slots of bxyz
    Meta m;
    int32_t* cnt;        // per warp unit: sent candidates
    int32_t* cntb;       // per block: sent candidates
    int32_t* cntb_home;  // per block: sent home atoms
    int32_t* blk_off;    // per block: output offset in the pulse's region
    const float* thr;  // thresholds of this pulse, by sender cell along d
    int nd, P, p, d, k, B;
    int nx, ny, nz;
    float Ld;
    // corner pruning (prune != 0)
    int prune;
    int nmax;
    double rc2;           // rc * rc in double, rc as fp32
    const double* faces;  // lower faces [3][nmax], then upper faces [3][nmax]
};

// Corner pruning: distance of a candidate (coordinates v, forwarding dims m)
// of sender cell c to the receiver's home box, over the pulse's dim d and the
// dims the slot was received across, below rc?  Double precision with
// explicit round-to-nearest operations (no contraction), d's term first, then
// ascending dims.
__device__ __forceinline__ bool corner_within(const PulseArgs& a, const int c[3], const float v[3],
                                              unsigned m) {
    double t = __dsub_rn((double)v[a.d], a.faces[a.d * a.nmax + c[a.d]]);
    t = t > 0.0 ? t : 0.0;
    double r2 = __dmul_rn(t, t);
#pragma unroll
    for (int e = 0; e < 3; e++) {
        if (e == a.d || !((m >> e) & 1u)) continue;
        double u = __dsub_rn((double)v[e], a.faces[(3 + e) * a.nmax + c[e]]);
        u = u > 0.0 ? u : 0.0;
        r2 = __dadd_rn(r2, __dmul_rn(u, u));
    }
    return r2 < a.rc2;
}

struct Locator {
    int64_t oo[HALO_MAX_PULSES + 1];
    int64_t rp[HALO_MAX_PULSES];
    int64_t hstart;
};

// Build-buffer slot of local index i of the block's sender (i < oo[p]).
__device__ __forceinline__ int64_t locate(const Locator& L, int p, int64_t i) {
    if (i < L.oo[0]) return L.hstart + i;
    int q = p - 1;
    while (q > 0 && i < L.oo[q]) q--;
    return L.rp[q] + (i - L.oo[q]);
}

__device__ __forceinline__ void load_locator(Locator& L, const PulseArgs& a, int s) {
    const int64_t* oo = a.m.own_off + (int64_t)s * (a.P + 1);
    const int64_t* rp = a.m.recv_pos + (int64_t)s * a.P;
    for (int q = threadIdx.x; q <= a.p; q += blockDim.x) L.oo[q] = oo[q];
    for (int q = threadIdx.x; q < a.p; q += blockDim.x) L.rp[q] = rp[q];
    if (threadIdx.x == 0) L.hstart = a.m.hstart[s];
    __syncthreads();
}

// Warp-granular work: block b of sender s has kPulseWarps warps, and warp w
// takes unit u = b * kPulseWarps + w of the B * kPulseWarps contiguous, equal
// parts of the candidate range (so the units, in order, cover it in order).
constexpr int kPulseWarps = kThreads / 32;

__device__ __forceinline__ void unit_range(const Locator& L, const PulseArgs& a, int u,
                                           int64_t* lo, int64_t* hi) {
    const int64_t c0 = (a.k == 0) ? 0 : L.oo[a.p - 1];
    const int64_t c1 = L.oo[a.p];
    const int64_t len = c1 - c0;
    const int64_t units = (int64_t)a.B * kPulseWarps;
    *lo = c0 + len * u / units;
    *hi = c0 + len * (u + 1) / units;
}

// Is candidate slot v (coordinates, forwarding dims in w) sent by this pulse?
__device__ __forceinline__ bool pulse_selects(const PulseArgs& a, const int cell[3], float thr,
                                              const float4& v) {
    const float vd = a.d == 0 ? v.x : (a.d == 1 ? v.y : v.z);
    if (!(vd < thr)) return false;
    if (!a.prune) return true;
    const float c[3] = {v.x, v.y, v.z};
    return corner_within(a, cell, c, (unsigned)__float_as_int(v.w));
}

// Output offsets of the pulse from the block counts, run by the last count
// block: blk_off[s*B + b] = the exclusive prefix of the block counts over all
// senders' blocks (relative to the pulse's region); per sender s its send
// size, split and output start; the receiver's slice position and local
// offsets.  Rounds of whole senders, eight block counts per thread; counts
// are read through L2 (other blocks wrote them in this launch).
constexpr int kOffsetSenders = 1024;  // senders per round of pulse_offsets

__device__ void pulse_offsets(const PulseArgs& a, int32_t* dsnd, int32_t* dspl) {
    constexpr int EPT = 8;
    const int64_t B = a.B;
    const int64_t dpr = min((int64_t)kOffsetSenders, max((int64_t)1, EPT * kThreads / B));
    const int64_t R = a.m.region[a.p];
    int64_t carry = 0;
    for (int64_t s0 = 0; s0 < a.nd; s0 += dpr) {
        const int64_t ns = min(dpr, (int64_t)a.nd - s0);
        const int64_t e0 = s0 * B, e1 = (s0 + ns) * B;  // this round's entries
        const int64_t i0 = e0 + EPT * threadIdx.x;
        for (int64_t j = threadIdx.x; j < dpr; j += kThreads) dsnd[j] = dspl[j] = 0;
        int32_t c[EPT], h[EPT];
        int64_t cs = 0;
#pragma unroll
        for (int k = 0; k < EPT; k++) {
            const bool in = i0 + k < e1;
            c[k] = in ? __ldcg(a.cntb + i0 + k) : 0;
            h[k] = in ? __ldcg(a.cntb_home + i0 + k) : 0;
            cs += c[k];
        }
        __syncthreads();
        int64_t tot;
        int64_t run = carry + block_exclusive_scan<kThreads>(cs, &tot);
#pragma unroll
        for (int k = 0; k < EPT; k++) {
            if (i0 + k < e1) {
                a.blk_off[i0 + k] = (int32_t)run;
                const int64_t j = (i0 + k) / B - s0;
                atomicAdd(&dsnd[j], c[k]);
                atomicAdd(&dspl[j], h[k]);
            }
            run += c[k];
        }
        __syncthreads();
        for (int64_t j = threadIdx.x; j < ns; j += kThreads) {
            const int s = (int)(s0 + j);
            const int64_t snd = dsnd[j], spl = dspl[j];
            const int64_t G = a.blk_off[(int64_t)s * B];
            const int64_t sp = (int64_t)s * a.P + a.p;
            a.m.send[sp] = snd;
            a.m.split[sp] = spl;
            a.m.map_pos[sp] = R + G;
            int cc[3] = {s % a.nx, (s / a.nx) % a.ny, s / (a.nx * a.ny)};
            const int nd_d = a.d == 0 ? a.nx : (a.d == 1 ? a.ny : a.nz);
            cc[a.d] = (cc[a.d] - 1 + nd_d) % nd_d;
            const int r = cc[0] + a.nx * (cc[1] + a.ny * cc[2]);
            a.m.recv_pos[(int64_t)r * a.P + a.p] = R + G;
            a.m.own_off[(int64_t)r * (a.P + 1) + a.p + 1] =
                a.m.own_off[(int64_t)r * (a.P + 1) + a.p] + snd;
        }
        carry += tot;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        a.m.region[a.p + 1] = R + carry;
        if (R + carry > a.cap) a.m.flags[0] = 1;
    }
}

// Per unit: how many candidates the pulse sends, and how many of them are
// home atoms (the split).  Each warp counts its unit 32 candidates at a time,
// U rounds' loads in flight.  The last block to finish (an atomic ticket in
// flags[3], reset for the next pulse) computes the offsets.
__global__ void __launch_bounds__(kThreads) pulse_count_kernel(PulseArgs a) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    __shared__ Locator L;
    const int s = blockIdx.y;
    load_locator(L, a, s);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int u0 = blockIdx.x * kPulseWarps + w;
    const int cs = cell_of(s, a.d, a.nx, a.ny);
    const float thr = a.thr[cs];
    const int cell[3] = {s % a.nx, (s / a.nx) % a.ny, s / (a.nx * a.ny)};
    int64_t lo, hi;
    unit_range(L, a, u0, &lo, &hi);
    const int64_t nh = L.oo[0];
    int c = 0, ch = 0;
    constexpr int U = 8;
    for (int64_t t0 = lo; t0 < hi; t0 += U * 32) {
        float4 v[U];
        bool in[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t i = t0 + u * 32 + lane;
            const int64_t pos = i < hi ? locate(L, a.p, i) : -1;
            in[u] = pos >= 0 && pos < a.cap;
            v[u] = in[u] ? a.bxyz[pos] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            const bool sel = in[u] && pulse_selects(a, cell, thr, v[u]);
            const unsigned bal = __ballot_sync(kFull, sel);
            c += __popc(bal);
            const int64_t i0 = t0 + u * 32;  // the round's first candidate
            if (i0 < nh) ch += __popc(bal & (nh - i0 >= 32 ? kFull : ((1u << (nh - i0)) - 1u)));
        }
    }
    // per warp (its offset within the block, for the write kernel) and per
    // block (for the offsets)
    __shared__ int32_t wc[kPulseWarps], wh[kPulseWarps];
    __shared__ int32_t dsnd[kOffsetSenders], dspl[kOffsetSenders];
    __shared__ int last;
    if (lane == 0) {
        a.cnt[(int64_t)s * a.B * kPulseWarps + u0] = c;
        wc[w] = c;
        wh[w] = ch;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int32_t tc = 0, th = 0;
        for (int q = 0; q < kPulseWarps; q++) {
            tc += wc[q];
            th += wh[q];
        }
        a.cntb[(int64_t)s * a.B + blockIdx.x] = tc;
        a.cntb_home[(int64_t)s * a.B + blockIdx.x] = th;
        __threadfence();
        unsigned long long* ticket = reinterpret_cast<unsigned long long*>(a.m.flags + 3);
        last = atomicAdd(ticket, 1ull) == (unsigned long long)gridDim.x * gridDim.y - 1;
        if (last) *ticket = 0;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    pulse_offsets(a, dsnd, dspl);
}

// Each warp writes its unit's sent candidates from the unit's scanned offset
// on, in candidate order (ranks from the round's ballot): no block barrier.
__global__ void __launch_bounds__(kThreads) pulse_write_kernel(PulseArgs a) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    __shared__ Locator L;
    const int s = blockIdx.y;
    load_locator(L, a, s);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int u0 = blockIdx.x * kPulseWarps + w;
    const int cs = cell_of(s, a.d, a.nx, a.ny);
    const float thr = a.thr[cs];
    const int cell[3] = {s % a.nx, (s / a.nx) % a.ny, s / (a.nx * a.ny)};
    float sh[3] = {0.0f, 0.0f, 0.0f};
    if (cs == 0) sh[a.d] = a.Ld;
    int64_t lo, hi;
    unit_range(L, a, u0, &lo, &hi);
    int64_t out = a.m.region[a.p] + a.blk_off[(int64_t)s * a.B + blockIdx.x];
    {
        const int32_t* wcnt = a.cnt + ((int64_t)s * a.B + blockIdx.x) * kPulseWarps;
        const int32_t v = lane < w ? wcnt[lane] : 0;
        out += __reduce_add_sync(kFull, (unsigned)v);
    }
    const unsigned lt = lanemask_lt();
    const unsigned bit = 1u << a.d;
    constexpr int U = 8;
    for (int64_t t0 = lo; t0 < hi; t0 += U * 32) {
        float4 v[U];
        bool in[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t i = t0 + u * 32 + lane;
            const int64_t pos = i < hi ? locate(L, a.p, i) : -1;
            in[u] = pos >= 0 && pos < a.cap;
            v[u] = in[u] ? a.bxyz[pos] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            const bool sel = in[u] && pulse_selects(a, cell, thr, v[u]);
            const unsigned bal = __ballot_sync(kFull, sel);
            if (sel) {
                const int64_t o = out + __popc(bal & lt);
                if (o >= a.N && o < a.cap) {
                    const unsigned m = (unsigned)__float_as_int(v[u].w);
                    a.maps[o - a.N] = (int32_t)(t0 + u * 32 + lane);
                    a.bxyz[o] = make_float4(v[u].x + sh[0], v[u].y + sh[1], v[u].z + sh[2],
                                            __int_as_float((int)(m | bit)));
                }
            }
            out += __popc(bal);
        }
    }
}

// ---- 3. finalize -----------------------------------------------------------------
// Pulse descriptors on the device, from the metadata: the fields of the
// host's copy of the plan (map offset, sender base, the halo slice's first
// dense slot in the receiver, sizes, the shift across the periodic boundary),
// so the kernels that read them can run before the host has its own copy.
struct SPArgs {
    int8_t dim[HALO_MAX_PULSES];
    float box[3];
    int nx, ny, nz, nd, P;
    int64_t n;
};

// One block: every domain's first dense slot (exclusive scan of the local
// counts).
__global__ void __launch_bounds__(1024) finalize_kernel(Meta m, int nd, int P) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    int64_t carry = 0;
    for (int D0 = 0; D0 < nd; D0 += 1024) {
        const int D = D0 + threadIdx.x;
        const int64_t v = D < nd ? m.own_off[(int64_t)D * (P + 1) + P] : 0;
        int64_t tot;
        const int64_t pre = block_exclusive_scan<1024>(v, &tot);
        if (D < nd) m.base[D] = carry + pre;
        carry += tot;
    }
}

// Block D: D's pulse descriptors (as sender) and, if host_meta is given (the
// host's mapped staging), its share of the metadata words for the host.
__global__ void sp_meta_kernel(Meta m, SPArgs a, SPDesc* __restrict__ out,
                               const int64_t* __restrict__ meta, int64_t meta_words,
                               int64_t* __restrict__ host_meta) {
    grid_launch_dependents();  // the next kernel may start; it waits for this one
    grid_dependency_wait();
    const int D = blockIdx.x;
    if (host_meta) {
        const int64_t w0 = meta_words * D / gridDim.x, w1 = meta_words * (D + 1) / gridDim.x;
        for (int64_t q = w0 + threadIdx.x; q < w1; q += blockDim.x) host_meta[q] = meta[q];
    }
    const int64_t b = m.base[D];
    const int P = a.P;
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        const int s = D;
        const int64_t i = (int64_t)s * P + p;
        const int d = a.dim[p];
        const int g[3] = {a.nx, a.ny, a.nz};
        int c[3] = {s % a.nx, (s / a.nx) % a.ny, s / (a.nx * a.ny)};
        const bool wrap = c[d] == 0;
        c[d] = (c[d] - 1 + g[d]) % g[d];
        const int r = c[0] + a.nx * (c[1] + a.ny * c[2]);
        SPDesc x;
        x.map_off = m.map_pos[i] - a.n;
        x.src_base = b;
        x.dst = m.base[r] + m.own_off[(int64_t)r * (P + 1) + p];
        x.send = (int32_t)m.send[i];
        x.split = (int32_t)m.split[i];
        x.s = s;
        x.r = r;
        x.p = p;
        x.pad = 0;
        x.shift[0] = x.shift[1] = x.shift[2] = 0.0f;
        if (wrap) x.shift[d] = a.box[d];
        x.pad2 = 0.0f;
        out[i] = x;
    }
}

int grow(float** p, int64_t* cap_have, int64_t need_slots) {
    if (*p && *cap_have >= need_slots) return HALO_OK;
    dev_free(*p);
    *cap_have = 0;
    HALO_TRY(dev_alloc(p, (size_t)need_slots * 4));  // one float4 per slot
    *cap_have = need_slots;
    return HALO_OK;
}

}  // namespace

int device_exclusive_scan(const int32_t* in, int32_t* out, int64_t n, int32_t* tmp,
                          cudaStream_t st) {
    const int64_t nb = (n + kScanTile - 1) / kScanTile;
    if (nb == 0) return HALO_OK;
    HALO_CUDA(launch_dependent_shm(scan_reduce_kernel, dim3((unsigned)nb), dim3(kThreads), 0, st, in, n, tmp));
    HALO_CUDA(launch_dependent_shm(scan_top_kernel, dim3(1), dim3(1024), 0, st, tmp, nb));
    HALO_CUDA(launch_dependent_shm(scan_down_kernel, dim3((unsigned)nb), dim3(kThreads), 0, st, in, out, n,
                                   (const int32_t*)tmp));
    return HALO_OK;
}

void free_build(halo_plan* pl) {
    dev_free(pl->d_bxyz);
    dev_free(pl->d_maps);
    dev_free(pl->d_home_gid);
    dev_free(pl->d_counts);
    dev_free(pl->d_scan_tmp);
    dev_free(pl->d_meta);
    dev_free(pl->d_pulse_scratch);
    dev_free(pl->d_thr);
    dev_free(pl->d_faces);
    pl->cap_slots = 0;
    pl->n_alloc_atoms = 0;
    pl->counts_cap = 0;
    pl->scan_tmp_cap = 0;
    pl->meta_bytes = 0;
}

DomainTables domain_tables(const halo_plan* pl) {
    const Meta m = meta_ptrs(pl->d_meta, pl->n_dom, pl->P);
    return DomainTables{m.n_home, m.hstart, m.base, m.own_off};
}

int build_plan(halo_plan* pl, const float* coords, const int32_t* dom, int64_t n,
               cudaStream_t st) {
    const int nd = pl->n_dom, P = pl->P;
    // home partition.  Tiled: tiles of T atoms, each ranked in shared memory
    // by a scatter block of kScatterThreads / 32 warp sub-tiles; T is the
    // largest of 8192 .. 1024 with two scatter blocks per SM (the per-warp
    // histograms must fit 48 KB, and a block scans the domains two per
    // thread).  Measured on the 3M-atom system (T = 4096,
    // 256 threads): rebuild 0.59 ms against 0.60 at T = 2048 (three blocks
    // per SM) and 0.60 at T = 8192 (one); 512 threads, 5 us less.  Otherwise
    // the direct
    // scatter: W warps per block (their histograms share 48 KB of shared
    // memory), one block tile of W * kHistTile atoms per block.
    int tileT = 0;
    size_t tile_smem = 0;
    if ((size_t)(kScatterThreads / 32) * nd * sizeof(int32_t) <= 48 * 1024 && nd <= 2 * kScatterThreads) {
        int optin = 0, per_sm = 0;
        HALO_CUDA(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, pl->dev));
        HALO_CUDA(cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, pl->dev));
        for (int T : {8192, 4096, 2048, 1024}) {
            const size_t need = tile_scatter_smem(kScatterThreads / 32, nd, T);
            if (need <= (size_t)optin && 2 * (need + 1024) <= (size_t)per_sm) {
                tileT = T;
                tile_smem = need;
                break;
            }
        }
        if (tileT > 0)
            HALO_CUDA(cudaFuncSetAttribute(home_scatter_tile_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tile_smem));
    }
    const int wpb = tileT > 0 ? kThreads / 32
                              : (int)std::min<int64_t>(8, std::max<int64_t>(1, (48 * 1024) / ((int64_t)nd * 4)));
    const int wtile = tileT > 0 ? tileT / wpb : kHistTile;
    const size_t hist_smem = (size_t)wpb * nd * sizeof(int32_t);
    const int64_t nbt = (n + (int64_t)wpb * wtile - 1) / ((int64_t)wpb * wtile);
    const unsigned hist_blocks = (unsigned)std::max<int64_t>(nbt, 1);

    // --- buffers that depend on N
    if (n > pl->n_alloc_atoms) {
        dev_free(pl->d_home_gid);
        pl->n_alloc_atoms = 0;
        HALO_TRY(dev_alloc(&pl->d_home_gid, (size_t)n));
        pl->n_alloc_atoms = n;
    }
    const int64_t ncount = (int64_t)nd * nbt;
    // block-tile counts, their scanned offsets, then (direct scatter) every
    // warp's counts (block-major: [block tile][warp][domain])
    const int64_t nwc = tileT > 0 ? 0 : (int64_t)nd * nbt * wpb;
    if (2 * ncount + nwc > pl->counts_cap) {
        dev_free(pl->d_counts);
        pl->counts_cap = 0;
        HALO_TRY(dev_alloc(&pl->d_counts, (size_t)(2 * ncount + nwc)));
        pl->counts_cap = 2 * ncount + nwc;
    }
    const int64_t nsum = std::max<int64_t>((ncount + kScanTile - 1) / kScanTile, 1);
    if (nsum > pl->scan_tmp_cap) {
        dev_free(pl->d_scan_tmp);
        pl->scan_tmp_cap = 0;
        HALO_TRY(dev_alloc(&pl->d_scan_tmp, (size_t)nsum));
        pl->scan_tmp_cap = nsum;
    }
    const size_t mbytes = meta_count(nd, P) * sizeof(int64_t);
    if (mbytes > pl->meta_bytes) {
        dev_free(pl->d_meta);
        pl->meta_bytes = 0;
        HALO_TRY(dev_alloc((char**)&pl->d_meta, mbytes));
        pl->meta_bytes = mbytes;
    }
    // blocks per sender domain in the pulse kernels: enough blocks to fill the
    // GPU, but at least ~256 candidates per block
    {
        const int64_t per_dom = n / nd + 1;
        int64_t B = std::max<int64_t>(1, (int64_t)8 * pl->num_sms / nd);
        B = std::min<int64_t>(B, std::max<int64_t>(1, per_dom / 256));
        B = std::min<int64_t>(B, 64);
        if (B != pl->build_blocks_per_domain || !pl->d_pulse_scratch) {
            dev_free(pl->d_pulse_scratch);
            HALO_TRY(dev_alloc(&pl->d_pulse_scratch, (size_t)nd * B * (kPulseWarps + 3)));
            pl->build_blocks_per_domain = (int)B;
        }
    }
    const int B = pl->build_blocks_per_domain;
    // thresholds: fl32(c * L_d / n_d + rc), evaluated in double, per pulse and sender cell
    if (!pl->d_thr && P > 0) {
        const int nmax = std::max(pl->grid[0], std::max(pl->grid[1], pl->grid[2]));
        std::vector<float> thr((size_t)P * nmax, 0.0f);
        for (int p = 0; p < P; p++) {
            const int d = pl->pulse_dim[p];
            for (int c = 0; c < pl->grid[d]; c++)
                thr[(size_t)p * nmax + c] =
                    (float)((double)c * (double)pl->box[d] / (double)pl->grid[d] + (double)pl->rc);
        }
        HALO_TRY(dev_alloc(&pl->d_thr, thr.size()));
        HALO_CUDA(cudaMemcpy(pl->d_thr, thr.data(), thr.size() * sizeof(float),
                             cudaMemcpyHostToDevice));
    }
    const int nmax = std::max(pl->grid[0], std::max(pl->grid[1], pl->grid[2]));
    const bool prune = (pl->flags & HALO_SETUP_PRUNE_CORNERS) != 0;
    // corner pruning: faces c * L_d / n_d (lower) and (c + 1) * L_d / n_d (upper), in double
    if (prune && !pl->d_faces) {
        std::vector<double> faces((size_t)6 * nmax, 0.0);
        for (int d = 0; d < 3; d++)
            for (int c = 0; c < pl->grid[d]; c++) {
                faces[(size_t)d * nmax + c] = (double)c * (double)pl->box[d] / (double)pl->grid[d];
                faces[(size_t)(3 + d) * nmax + c] =
                    (double)(c + 1) * (double)pl->box[d] / (double)pl->grid[d];
            }
        HALO_TRY(dev_alloc(&pl->d_faces, faces.size()));
        HALO_CUDA(cudaMemcpy(pl->d_faces, faces.data(), faces.size() * sizeof(double),
                             cudaMemcpyHostToDevice));
    }

    // capacity estimate: each decomposed dim widens a domain by rc
    double grow_f = 1.0;
    for (int d = 0; d < 3; d++)
        if (pl->grid[d] > 1) grow_f *= 1.0 + (double)pl->rc / ((double)pl->box[d] / pl->grid[d]);
    int64_t want = n + (int64_t)ceil((double)n * (grow_f - 1.0) * 1.15) + (int64_t)256 * nd * P + 1024;
    want = std::max(want, pl->cap_slots);
    if (pl->debug_capacity > 0) {
        // test hook: start from the given capacity (the retry below grows it)
        dev_free(pl->d_bxyz);
        dev_free(pl->d_maps);
        pl->cap_slots = 0;
        want = std::max<int64_t>(pl->debug_capacity, n + 1);  // the home region always fits
        pl->debug_capacity = 0;
    }
    pl->build_attempts = 0;


    const Meta m = meta_ptrs(pl->d_meta, nd, P);
    HALO_TRY(dev_reserve(&pl->d_sp, &pl->cap_sp, (int64_t)nd * P));
    SPArgs spa;
    for (int p = 0; p < HALO_MAX_PULSES; p++) spa.dim[p] = (int8_t)(p < P ? pl->pulse_dim[p] : 0);
    for (int d = 0; d < 3; d++) spa.box[d] = pl->box[d];
    spa.nx = pl->grid[0];
    spa.ny = pl->grid[1];
    spa.nz = pl->grid[2];
    spa.nd = nd;
    spa.P = P;
    spa.n = n;
    void* hstage = nullptr;
    HALO_TRY(host_stage(pl, mbytes, &hstage));
    int64_t* hm = static_cast<int64_t*>(hstage);
    const Meta h = meta_ptrs(hm, nd, P);


    for (int attempt = 0; attempt < 6; attempt++) {
        pl->build_attempts = attempt + 1;
        if (want > pl->cap_slots) {
            int64_t have = pl->cap_slots;
            HALO_TRY(grow(&pl->d_bxyz, &have, want));
            // maps[slot - N] for slots in [N, cap): sized by cap so that any N fits
            dev_free(pl->d_maps);
            HALO_TRY(dev_alloc(&pl->d_maps, (size_t)want));
            pl->cap_slots = want;
        } else if (!pl->d_maps) {
            HALO_TRY(dev_alloc(&pl->d_maps, (size_t)pl->cap_slots));
        }
        HALO_CUDA(cudaMemsetAsync(pl->d_meta, 0, mbytes, st));
        // 1. home partition
        int32_t* wcounts = tileT > 0 ? nullptr : pl->d_counts + 2 * ncount;
        HALO_CUDA(launch_dependent_shm(home_hist_kernel, dim3(hist_blocks), dim3(wpb * 32), hist_smem, st,
                                       dom, n, nd, nbt, wtile, tileT > 0 ? 1 : 0, pl->d_counts, wcounts,
                                       m.flags));
        int32_t* offs = pl->d_counts + ncount;
        if (tileT > 0) {
            // column prefixes (tile-major, so each scatter block reads its
            // domains' starts contiguously) and the per-domain home metadata
            HALO_CUDA(launch_dependent_shm(home_colscan_kernel, dim3((unsigned)((nd + 31) / 32)), dim3(1024),
                                           0, st, (const int32_t*)pl->d_counts, nbt, nd, P, n, offs, m));
            const int vec = ((uintptr_t)coords % 16 == 0 && (uintptr_t)dom % 16 == 0) ? 1 : 0;
            HALO_CUDA(launch_dependent_shm(home_scatter_tile_kernel, dim3(hist_blocks), dim3(kScatterThreads),
                                           tile_smem, st, coords, dom, n, nd, tileT, vec,
                                           (const int32_t*)offs, (const int64_t*)m.hstart, pl->d_home_gid,
                                           reinterpret_cast<float4*>(pl->d_bxyz)));
        } else {
            HALO_TRY(device_exclusive_scan(pl->d_counts, offs, ncount, pl->d_scan_tmp, st));
            home_scatter_kernel<<<hist_blocks, wpb * 32, hist_smem, st>>>(
                coords, dom, n, nd, nbt, offs, wcounts, pl->d_home_gid,
                reinterpret_cast<float4*>(pl->d_bxyz));
            home_meta_kernel<<<(nd + 255) / 256, 256, 0, st>>>(offs, nbt, n, nd, P, m);
        }
        HALO_CUDA(cudaGetLastError());
        // 2. pulses in global order
        for (int p = 0; p < P; p++) {
            PulseArgs a;
            a.bxyz = reinterpret_cast<float4*>(pl->d_bxyz);
            a.maps = pl->d_maps;
            a.N = n;
            a.cap = pl->cap_slots;
            a.m = m;
            a.cnt = pl->d_pulse_scratch;
            a.cntb = a.cnt + (size_t)nd * B * kPulseWarps;
            a.cntb_home = a.cntb + (size_t)nd * B;
            a.blk_off = a.cntb_home + (size_t)nd * B;
            a.thr = pl->d_thr + (size_t)p * nmax;
            a.nd = nd;
            a.P = P;
            a.p = p;
            a.d = pl->pulse_dim[p];
            a.k = pl->pulse_k[p];
            a.B = B;
            a.nx = pl->grid[0];
            a.ny = pl->grid[1];
            a.nz = pl->grid[2];
            a.Ld = pl->box[a.d];
            a.prune = prune ? 1 : 0;
            a.nmax = nmax;
            a.rc2 = (double)pl->rc * (double)pl->rc;
            a.faces = pl->d_faces;
            dim3 g((unsigned)B, (unsigned)nd);
            HALO_CUDA(launch_dependent_shm(pulse_count_kernel, g, dim3(kThreads), 0, st, a));
            HALO_CUDA(launch_dependent_shm(pulse_write_kernel, g, dim3(kThreads), 0, st, a));
        }
        // 3. dense layout
        HALO_CUDA(launch_dependent_shm(finalize_kernel, dim3(1), dim3(1024), 0, st, m, nd, P));
        // the metadata comes back through the mapped staging (written by the
        // home slot kernel), else with a copy
        int64_t* host_meta = static_cast<int64_t*>(pl->h_stage_dev);
        HALO_CUDA(launch_dependent_shm(sp_meta_kernel, dim3(nd), dim3(256), 0, st, m, spa,
                                       pl->d_sp, reinterpret_cast<const int64_t*>(pl->d_meta),
                                       (int64_t)(mbytes / sizeof(int64_t)), host_meta));
        HALO_CUDA(cudaGetLastError());
        if (!host_meta) HALO_CUDA(cudaMemcpyAsync(hm, pl->d_meta, mbytes, cudaMemcpyDeviceToHost, st));
        HALO_CUDA(cudaStreamSynchronize(st));
        if (h.flags[1]) return HALO_EDOMAIN;
        if (!h.flags[0]) break;
        if (attempt == 5) return HALO_ECAPACITY;
        want = std::max<int64_t>(2 * pl->cap_slots, h.region[P] + h.region[P] / 4);
    }

    // host copy of the plan
    pl->n_atoms = n;
    pl->n_home.assign(nd, 0);
    pl->n_local.assign(nd, 0);
    pl->base.assign(nd, 0);
    pl->own_off.assign((size_t)nd * (P + 1), 0);
    pl->send.assign((size_t)nd * P, 0);
    pl->split.assign((size_t)nd * P, 0);
    pl->map_off.assign((size_t)nd * P, 0);
    int64_t tot = 0;
    for (int D = 0; D < nd; D++) {
        pl->n_home[D] = (int32_t)h.n_home[D];
        pl->n_local[D] = (int32_t)h.own_off[(size_t)D * (P + 1) + P];
        pl->base[D] = h.base[D];
        for (int q = 0; q <= P; q++)
            pl->own_off[(size_t)D * (P + 1) + q] = (int32_t)h.own_off[(size_t)D * (P + 1) + q];
        tot += pl->n_local[D];
    }
    pl->max_chunks.assign((size_t)std::max(P, 1), 0);
    for (size_t i = 0; i < (size_t)nd * P; i++) {
        pl->send[i] = (int32_t)h.send[i];
        pl->split[i] = (int32_t)h.split[i];
        pl->map_off[i] = h.map_pos[i] - n;
        const int p = (int)(i % P);
        pl->max_chunks[p] = std::max(pl->max_chunks[p], (pl->send[i] + kThreads - 1) / kThreads);
    }
    pl->n_local_total = tot;
    pl->n_halo_total = tot - n;
    if (P > 0 && h.region[P] - n != pl->n_halo_total) return HALO_ECAPACITY;
    return HALO_OK;
}

}  // namespace halo
