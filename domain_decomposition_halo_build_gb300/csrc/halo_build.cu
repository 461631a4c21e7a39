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
//      shared histograms), exclusive scan, stable scatter (warp match +
//      running per-domain counters) -> every domain's home atoms in input
//      order, in a home-compact region;
//   2. per pulse: count kernel (predicate per candidate, with the optional
//      corner test), scan kernel (block offsets, sizes, receiver offsets),
//      write kernel (stable block-wide ballot compaction -> ascending index
//      map + the new halo coordinates);
//   3. finalize: dense bases, home slot -> dense slot map; one D2H copy of the
//      metadata.
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


// ---- 1. home partition ------------------------------------------------------------
// A block of W warps covers the block tile b of W * kHistTile atoms; warp w
// its sub-tile [(b*W + w)*kHistTile, ... + kHistTile).  Each warp counts its
// sub-tile into its own shared histogram (shared-memory atomics); the block
// writes one count per domain, counts[D*nbt + b] (domain-major, so one
// exclusive scan gives every (domain, block tile) start), and every warp's
// counts, wcounts[(b*W + w)*nd + D] (contiguous per block, for the scatter).
__global__ void home_hist_kernel(const int32_t* __restrict__ dom, int64_t n, int nd, int64_t nbt,
                                 int32_t* __restrict__ counts, int32_t* __restrict__ wcounts,
                                 int64_t* __restrict__ flags) {
    extern __shared__ int32_t sh[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int W = blockDim.x >> 5;
    int32_t* h = sh + (size_t)warp * nd;
    for (int i = lane; i < nd; i += 32) h[i] = 0;
    __syncwarp();
    const int64_t a0 = ((int64_t)blockIdx.x * W + warp) * kHistTile;
    bool bad = false;
    // eight coalesced loads in flight per lane, then their counts
    constexpr int U = 8;
    for (int it = 0; it < kHistTile / 32; it += U) {
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
    int32_t* wc = wcounts + (int64_t)blockIdx.x * W * nd;
    for (int i = threadIdx.x; i < W * nd; i += blockDim.x) wc[i] = sh[i];
    for (int d = threadIdx.x; d < nd; d += blockDim.x) {
        int32_t t = 0;
        for (int w = 0; w < W; w++) t += sh[(size_t)w * nd + d];
        counts[(int64_t)d * nbt + blockIdx.x] = t;
    }
}

// Stable scatter: every warp's start per domain is its block tile's start
// plus the counts of the warps before it; then each warp visits its atoms in
// input order, and within 32 atoms the rank among equal domain ids comes from
// the warp match mask.
__global__ void home_scatter_kernel(const float* __restrict__ xyz, const int32_t* __restrict__ dom,
                                    int64_t n, int nd, int64_t nbt,
                                    const int32_t* __restrict__ offs,
                                    const int32_t* __restrict__ wcounts,
                                    int32_t* __restrict__ home_gid, float4* __restrict__ bxyz) {
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
            const unsigned peers = __match_any_sync(kFull, d[u]);
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

// The same stable scatter through shared memory: the block first places its
// tile's atoms in domain order in shared memory (warp by warp, 32 atoms at a
// time, ranks from the warp match mask, so the order within a domain stays
// the input order), then writes each domain's run of the tile contiguously.
// The global stores then fill whole sectors; scattered one atom per domain,
// each partly written sector had to be fetched from DRAM first.
__host__ __device__ inline size_t staged_scatter_smem(int W, int nd) {
    const size_t head = ((size_t)W * nd + 2 * (size_t)nd + 1) * sizeof(int32_t);
    const size_t T = (size_t)W * kHistTile;
    return ((head + 15) & ~(size_t)15) + T * (sizeof(float4) + sizeof(int32_t) + sizeof(int16_t));
}

__global__ void home_scatter_staged_kernel(const float* __restrict__ xyz,
                                           const int32_t* __restrict__ dom, int64_t n, int nd,
                                           int64_t nbt, const int32_t* __restrict__ offs,
                                           const int32_t* __restrict__ wcounts,
                                           int32_t* __restrict__ home_gid, float4* __restrict__ bxyz) {
    extern __shared__ __align__(16) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int W = blockDim.x >> 5;
    const int T = W * kHistTile;
    int32_t* wpos = reinterpret_cast<int32_t*>(smem);  // W * nd: next sorted position, per warp and domain
    int32_t* lstart = wpos + (size_t)W * nd;           // nd + 1: first sorted position of each domain
    int32_t* gstart = lstart + nd + 1;                 // nd: the domain run's first home-compact slot
    const size_t head = ((size_t)W * nd + 2 * (size_t)nd + 1) * sizeof(int32_t);
    float4* st_xyz = reinterpret_cast<float4*>(smem + ((head + 15) & ~(size_t)15));
    int32_t* st_gid = reinterpret_cast<int32_t*>(st_xyz + T);
    int16_t* st_dom = reinterpret_cast<int16_t*>(st_gid + T);
    const int32_t* wc = wcounts + (int64_t)blockIdx.x * W * nd;
    for (int d = threadIdx.x; d < nd; d += blockDim.x) {
        int32_t t = 0;
        for (int w = 0; w < W; w++) t += wc[(size_t)w * nd + d];
        lstart[d] = t;
        gstart[d] = offs[(int64_t)d * nbt + blockIdx.x];
    }
    __syncthreads();
    // exclusive scan of the per-domain counts (the first warp, 32 at a time)
    if (warp == 0) {
        int32_t carry = 0;
        for (int d0 = 0; d0 < nd; d0 += 32) {
            const int d = d0 + lane;
            const int32_t v = d < nd ? lstart[d] : 0;
            int32_t x = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t y = __shfl_up_sync(kFull, x, o);
                if (lane >= o) x += y;
            }
            if (d < nd) lstart[d] = carry + x - v;
            carry += __shfl_sync(kFull, x, 31);
        }
        if (lane == 0) lstart[nd] = carry;
    }
    __syncthreads();
    for (int d = threadIdx.x; d < nd; d += blockDim.x) {
        int32_t acc = lstart[d];
        for (int w = 0; w < W; w++) {
            wpos[(size_t)w * nd + d] = acc;
            acc += wc[(size_t)w * nd + d];
        }
    }
    __syncthreads();
    int32_t* run = wpos + (size_t)warp * nd;
    const int64_t a0 = ((int64_t)blockIdx.x * W + warp) * kHistTile;
    const unsigned lt = lanemask_lt();
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
            const unsigned peers = __match_any_sync(kFull, d[u]);
            if (d[u] >= 0) {
                const int pos = run[d[u]] + __popc(peers & lt);
                st_xyz[pos] = make_float4(c[u][0], c[u][1], c[u][2], __int_as_float(0));
                st_gid[pos] = (int32_t)a;
                st_dom[pos] = (int16_t)d[u];
            }
            __syncwarp();
            if (d[u] >= 0 && lane == __ffs(peers) - 1) run[d[u]] += __popc(peers);
            __syncwarp();
        }
    }
    __syncthreads();
    // every domain's run of the tile, contiguous in the home-compact region
    const int total = lstart[nd];
    for (int i = threadIdx.x; i < total; i += blockDim.x) {
        const int dd = st_dom[i];
        const int64_t g = (int64_t)gstart[dd] + (i - lstart[dd]);
        bxyz[g] = st_xyz[i];
        home_gid[g] = st_gid[i];
    }
}

// ---- generic int32 exclusive scan (three launches) ---------------------------------
__global__ void scan_reduce_kernel(const int32_t* __restrict__ in, int64_t n,
                                   int32_t* __restrict__ sums) {
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
    int32_t* cnt;
    int32_t* cnt_home;
    int32_t* blk_off;
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

__device__ __forceinline__ void sub_range(const Locator& L, const PulseArgs& a, int b,
                                          int64_t* lo, int64_t* hi) {
    const int64_t c0 = (a.k == 0) ? 0 : L.oo[a.p - 1];
    const int64_t c1 = L.oo[a.p];
    const int64_t len = c1 - c0;
    *lo = c0 + len * b / a.B;
    *hi = c0 + len * (b + 1) / a.B;
}

__global__ void __launch_bounds__(kThreads) pulse_count_kernel(PulseArgs a) {
    __shared__ Locator L;
    const int s = blockIdx.y, b = blockIdx.x;
    load_locator(L, a, s);
    const int cs = cell_of(s, a.d, a.nx, a.ny);
    const float thr = a.thr[cs];
    const int cell[3] = {s % a.nx, (s / a.nx) % a.ny, s / (a.nx * a.ny)};
    int64_t lo, hi;
    sub_range(L, a, b, &lo, &hi);
    const int64_t nh = L.oo[0];
    int64_t c = 0, ch = 0;
    // four candidates per thread and step, their loads issued together
    constexpr int U = 4;
    for (int64_t i0 = lo + threadIdx.x; i0 < hi; i0 += U * kThreads) {
        float4 slot[U];
        bool in[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t i = i0 + u * kThreads;
            const int64_t pos = i < hi ? locate(L, a.p, i) : -1;
            in[u] = pos >= 0 && pos < a.cap;
            slot[u] = in[u] ? a.bxyz[pos] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            if (!in[u]) continue;
            const float vd = a.d == 0 ? slot[u].x : (a.d == 1 ? slot[u].y : slot[u].z);
            if (vd < thr) {
                if (a.prune) {
                    const float v[3] = {slot[u].x, slot[u].y, slot[u].z};
                    if (!corner_within(a, cell, v, (unsigned)__float_as_int(slot[u].w))) continue;
                }
                c++;
                if (i0 + u * kThreads < nh) ch++;
            }
        }
    }
    int64_t tc, th;
    block_exclusive_scan<kThreads>(c, &tc);
    block_exclusive_scan<kThreads>(ch, &th);
    if (threadIdx.x == 0) {
        a.cnt[(int64_t)s * a.B + b] = (int32_t)tc;
        a.cnt_home[(int64_t)s * a.B + b] = (int32_t)th;
    }
}

__global__ void __launch_bounds__(1024) pulse_scan_kernel(PulseArgs a) {
    const int64_t M = (int64_t)a.nd * a.B;
    int64_t carry = 0;
    for (int64_t b0 = 0; b0 < M; b0 += 1024) {
        const int64_t i = b0 + threadIdx.x;
        const int64_t v = i < M ? a.cnt[i] : 0;
        int64_t tot;
        const int64_t pre = block_exclusive_scan<1024>(v, &tot);
        if (i < M) a.blk_off[i] = (int32_t)(carry + pre);
        carry += tot;
    }
    __syncthreads();
    const int64_t R = a.m.region[a.p];
    for (int s = threadIdx.x; s < a.nd; s += blockDim.x) {
        int64_t snd = 0, spl = 0;
        for (int b = 0; b < a.B; b++) {
            snd += a.cnt[(int64_t)s * a.B + b];
            spl += a.cnt_home[(int64_t)s * a.B + b];
        }
        const int64_t G = a.blk_off[(int64_t)s * a.B];
        const int64_t sp = (int64_t)s * a.P + a.p;
        a.m.send[sp] = snd;
        a.m.split[sp] = spl;
        a.m.map_pos[sp] = R + G;
        int c[3] = {s % a.nx, (s / a.nx) % a.ny, s / (a.nx * a.ny)};
        const int nd_d = a.d == 0 ? a.nx : (a.d == 1 ? a.ny : a.nz);
        c[a.d] = (c[a.d] - 1 + nd_d) % nd_d;
        const int r = c[0] + a.nx * (c[1] + a.ny * c[2]);
        a.m.recv_pos[(int64_t)r * a.P + a.p] = R + G;
        a.m.own_off[(int64_t)r * (a.P + 1) + a.p + 1] =
            a.m.own_off[(int64_t)r * (a.P + 1) + a.p] + snd;
    }
    if (threadIdx.x == 0) {
        a.m.region[a.p + 1] = R + carry;
        if (R + carry > a.cap) a.m.flags[0] = 1;
    }
}

__global__ void __launch_bounds__(kThreads) pulse_write_kernel(PulseArgs a) {
    constexpr int U = 4;  // tiles of kThreads candidates per step
    __shared__ Locator L;
    __shared__ int wcnt[U][kThreads / 32];
    const int s = blockIdx.y, b = blockIdx.x;
    load_locator(L, a, s);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int cs = cell_of(s, a.d, a.nx, a.ny);
    const float thr = a.thr[cs];
    const int cell[3] = {s % a.nx, (s / a.nx) % a.ny, s / (a.nx * a.ny)};
    float sh[3] = {0.0f, 0.0f, 0.0f};
    if (cs == 0) sh[a.d] = a.Ld;
    int64_t lo, hi;
    sub_range(L, a, b, &lo, &hi);
    int64_t out = a.m.region[a.p] + a.blk_off[(int64_t)s * a.B + b];
    const unsigned lt = lanemask_lt();
    // U consecutive tiles per step: every candidate's load is issued first,
    // then the tiles are compacted in order (one barrier pair per step)
    for (int64_t t0 = lo; t0 < hi; t0 += U * kThreads) {
        float4 slot[U];
        bool sel[U];
        unsigned bal[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const int64_t i = t0 + u * kThreads + threadIdx.x;
            const int64_t pos = i < hi ? locate(L, a.p, i) : -1;
            sel[u] = pos >= 0 && pos < a.cap;
            slot[u] = sel[u] ? a.bxyz[pos] : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            if (sel[u]) {
                const float vd = a.d == 0 ? slot[u].x : (a.d == 1 ? slot[u].y : slot[u].z);
                sel[u] = vd < thr;
                if (sel[u] && a.prune) {
                    const float v[3] = {slot[u].x, slot[u].y, slot[u].z};
                    sel[u] = corner_within(a, cell, v, (unsigned)__float_as_int(slot[u].w));
                }
            }
            bal[u] = __ballot_sync(kFull, sel[u]);
            if (lane == 0) wcnt[u][warp] = __popc(bal[u]);
        }
        __syncthreads();
#pragma unroll
        for (int u = 0; u < U; u++) {
            int before = 0, total = 0;
#pragma unroll
            for (int w = 0; w < kThreads / 32; w++) {
                const int c = wcnt[u][w];
                before += (w < warp) ? c : 0;
                total += c;
            }
            if (sel[u]) {
                const int64_t o = out + before + __popc(bal[u] & lt);
                if (o >= a.N && o < a.cap) {
                    const unsigned m = (unsigned)__float_as_int(slot[u].w);
                    a.maps[o - a.N] = (int32_t)(t0 + u * kThreads + threadIdx.x);
                    a.bxyz[o] = make_float4(slot[u].x + sh[0], slot[u].y + sh[1], slot[u].z + sh[2],
                                            __int_as_float((int)(m | (1u << a.d))));
                }
            }
            out += total;
        }
        __syncthreads();
    }
}

// ---- 3. finalize -----------------------------------------------------------------
__global__ void __launch_bounds__(1024) finalize_kernel(Meta m, int nd, int P) {
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

__global__ void home_dst_kernel(Meta m, int64_t* __restrict__ home_dst) {
    const int D = blockIdx.x;
    const int64_t h0 = m.hstart[D], nh = m.n_home[D], b = m.base[D];
    for (int64_t j = threadIdx.x; j < nh; j += blockDim.x) home_dst[h0 + j] = b + j;
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
    scan_reduce_kernel<<<(unsigned)nb, kThreads, 0, st>>>(in, n, tmp);
    scan_top_kernel<<<1, 1024, 0, st>>>(tmp, nb);
    scan_down_kernel<<<(unsigned)nb, kThreads, 0, st>>>(in, out, n, tmp);
    return cuda_code(cudaGetLastError());
}

void free_build(halo_plan* pl) {
    dev_free(pl->d_bxyz);
    dev_free(pl->d_maps);
    dev_free(pl->d_home_gid);
    dev_free(pl->d_home_dst);
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

int build_plan(halo_plan* pl, const float* coords, const int32_t* dom, int64_t n,
               cudaStream_t st) {
    const int nd = pl->n_dom, P = pl->P;
    const int64_t ntiles = (n + kHistTile - 1) / kHistTile;
    // home partition: W warps per block (their histograms share 48 KB of
    // shared memory), one block tile of W * kHistTile atoms per block
    const int wpb = (int)std::min<int64_t>(8, std::max<int64_t>(1, (48 * 1024) / ((int64_t)nd * 4)));
    const size_t hist_smem = (size_t)wpb * nd * sizeof(int32_t);
    const int64_t nbt = (ntiles + wpb - 1) / wpb;
    const unsigned hist_blocks = (unsigned)std::max<int64_t>(nbt, 1);

    // --- buffers that depend on N
    if (n > pl->n_alloc_atoms) {
        dev_free(pl->d_home_gid);
        dev_free(pl->d_home_dst);
        pl->n_alloc_atoms = 0;
        HALO_TRY(dev_alloc(&pl->d_home_gid, (size_t)n));
        HALO_TRY(dev_alloc(&pl->d_home_dst, (size_t)n));
        pl->n_alloc_atoms = n;
    }
    const int64_t ncount = (int64_t)nd * nbt;
    // block-tile counts, their scanned offsets, then every warp's counts
    // (block-major: [block tile][warp][domain]) for the scatter
    const int64_t nwc = (int64_t)nd * nbt * wpb;
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
            HALO_TRY(dev_alloc(&pl->d_pulse_scratch, (size_t)3 * nd * B));
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

    // the home scatter sorts each tile in shared memory where the tile and
    // the per-domain tables fit (nd < 32768 for the int16 domain ids)
    size_t staged_smem = 0;
    {
        int optin = 0;
        HALO_CUDA(cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, pl->dev));
        const size_t need = staged_scatter_smem(wpb, nd);
        if (nd < 32768 && need <= (size_t)optin) {
            HALO_CUDA(cudaFuncSetAttribute(home_scatter_staged_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)need));
            staged_smem = need;
        }
    }

    const Meta m = meta_ptrs(pl->d_meta, nd, P);
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
        int32_t* wcounts = pl->d_counts + 2 * ncount;
        home_hist_kernel<<<hist_blocks, wpb * 32, hist_smem, st>>>(dom, n, nd, nbt,
                                                                  pl->d_counts, wcounts, m.flags);
        int32_t* offs = pl->d_counts + ncount;
        HALO_TRY(device_exclusive_scan(pl->d_counts, offs, ncount, pl->d_scan_tmp, st));
        if (staged_smem > 0)
            home_scatter_staged_kernel<<<hist_blocks, wpb * 32, staged_smem, st>>>(
                coords, dom, n, nd, nbt, offs, wcounts, pl->d_home_gid,
                reinterpret_cast<float4*>(pl->d_bxyz));
        else
            home_scatter_kernel<<<hist_blocks, wpb * 32, hist_smem, st>>>(
                coords, dom, n, nd, nbt, offs, wcounts, pl->d_home_gid,
                reinterpret_cast<float4*>(pl->d_bxyz));
        home_meta_kernel<<<(nd + 255) / 256, 256, 0, st>>>(offs, nbt, n, nd, P, m);
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
            a.cnt_home = pl->d_pulse_scratch + (size_t)nd * B;
            a.blk_off = pl->d_pulse_scratch + (size_t)2 * nd * B;
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
            pulse_count_kernel<<<g, kThreads, 0, st>>>(a);
            pulse_scan_kernel<<<1, 1024, 0, st>>>(a);
            pulse_write_kernel<<<g, kThreads, 0, st>>>(a);
        }
        // 3. dense layout
        finalize_kernel<<<1, 1024, 0, st>>>(m, nd, P);
        home_dst_kernel<<<nd, 256, 0, st>>>(m, pl->d_home_dst);
        HALO_CUDA(cudaGetLastError());
        HALO_CUDA(cudaMemcpyAsync(hm, pl->d_meta, mbytes, cudaMemcpyDeviceToHost, st));
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
    for (size_t i = 0; i < (size_t)nd * P; i++) {
        pl->send[i] = (int32_t)h.send[i];
        pl->split[i] = (int32_t)h.split[i];
        pl->map_off[i] = h.map_pos[i] - n;
    }
    pl->n_local_total = tot;
    pl->n_halo_total = tot - n;
    if (P > 0 && h.region[P] - n != pl->n_halo_total) return HALO_ECAPACITY;
    return HALO_OK;
}

}  // namespace halo
