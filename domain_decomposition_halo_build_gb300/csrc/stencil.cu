// stencil.cu -- the two-dimensional stencil halo workload (include/stencil.h).
//
// Page: "GPU-centric Communication on NVIDIA GPU Clusters with InfiniBand: A
// Case Study with OpenSHMEM", section "2D stencil mini-app": blocks of a
// matrix on a non-periodic 1-D or 2-D grid, each iteration a sweep of every
// block and an exchange of block edges with up to four neighbours; the page's
// fused kernel computes and sends in one launch.  All blocks share this GPU's
// memory, so a send is a store into the neighbour block's ghost cells.
//
// Kernels:
//   stencil_exchange_kernel: one thread per (block, side, 4 edge cells); rows
//     move as 16-byte vectors, columns as four strided floats.
//   stencil_sweep_kernel<FUSED>: a block of 128 threads covers 512 columns of
//     one matrix block over a band of 16 rows; every thread keeps the rows
//     above, at and below its 4 cells in registers and slides down the band,
//     so each input row is loaded once per band (plus the two rows around it);
//     the west and east neighbours of a 4-cell group come from the adjacent
//     lanes by shuffle, from memory only at warp and block edges.  FUSED also
//     stores each new edge value into the neighbouring block's ghost cell.
#include <cuda_runtime.h>
#include <stdint.h>

#include <new>

#include "stencil.h"

struct stencil_plan {
    int px = 0, py = 0, n = 0;
    int pitch = 0, rows = 0;
    int64_t tile_floats = 0, total_floats = 0;
};

namespace {

constexpr int kCol0 = 4;     // first block column of a tile row
constexpr int kQuads = 128;  // threads per sweep block, 4 cells each
constexpr int kBand = 16;    // rows per sweep block
constexpr int kExchThreads = 256;
constexpr unsigned kFull = 0xffffffffu;

struct Geo {
    int px, py, n, pitch;
    int64_t tile;  // floats per tile
};

__device__ __forceinline__ float4 ld4(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }

// Thread id -> (tile t, side s, group q of 4 edge cells), id < tiles * n.
// s: 0 first row -> ghost row below the block above; 1 last row -> ghost row
// above the block below; 2 first column -> east ghost column of the block on
// the left; 3 last column -> west ghost column of the block on the right.
// Reads are block cells, writes are ghost cells: the two sets are disjoint.
__global__ void __launch_bounds__(kExchThreads) stencil_exchange_kernel(float* f, Geo g,
                                                                        int64_t threads) {
    const int64_t id = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (id >= threads) return;
    const int nq = g.n / 4;
    const int q = (int)(id % nq);
    const int64_t ts = id / nq;
    const int s = (int)(ts & 3);
    const int t = (int)(ts >> 2);
    const int tx = t % g.px, ty = t / g.px;
    const float* me = f + (int64_t)t * g.tile;
    const int c = kCol0 + 4 * q;
    if (s == 0) {
        if (ty == 0) return;
        float* nb = f + (int64_t)(t - g.px) * g.tile;
        st4(nb + (int64_t)(g.n + 1) * g.pitch + c, ld4(me + (int64_t)g.pitch + c));
    } else if (s == 1) {
        if (ty == g.py - 1) return;
        float* nb = f + (int64_t)(t + g.px) * g.tile;
        st4(nb + c, ld4(me + (int64_t)g.n * g.pitch + c));
    } else if (s == 2) {
        if (tx == 0) return;
        float* nb = f + (int64_t)(t - 1) * g.tile;
        float v[4];
#pragma unroll
        for (int r = 0; r < 4; r++) v[r] = __ldg(me + (int64_t)(1 + 4 * q + r) * g.pitch + kCol0);
#pragma unroll
        for (int r = 0; r < 4; r++) nb[(int64_t)(1 + 4 * q + r) * g.pitch + kCol0 + g.n] = v[r];
    } else {
        if (tx == g.px - 1) return;
        float* nb = f + (int64_t)(t + 1) * g.tile;
        float v[4];
#pragma unroll
        for (int r = 0; r < 4; r++)
            v[r] = __ldg(me + (int64_t)(1 + 4 * q + r) * g.pitch + kCol0 + g.n - 1);
#pragma unroll
        for (int r = 0; r < 4; r++) nb[(int64_t)(1 + 4 * q + r) * g.pitch + kCol0 - 1] = v[r];
    }
}

// ((N + S) + (W + E)) * 0.25, one rounding per operation, no contraction.
__device__ __forceinline__ float jacobi(float n, float s, float w, float e) {
    return __fmul_rn(__fadd_rn(__fadd_rn(n, s), __fadd_rn(w, e)), 0.25f);
}

template <bool FUSED>
__global__ void __launch_bounds__(kQuads) stencil_sweep_kernel(const float* __restrict__ in,
                                                               float* out, Geo g) {
    const int nq = g.n / 4;
    const int q = blockIdx.x * kQuads + threadIdx.x;  // group of 4 columns
    const int r0 = 1 + blockIdx.y * kBand;             // first row of the band (<= n)
    const int r1 = min(r0 + kBand, g.n + 1);           // one past its last row
    const int t = blockIdx.z;
    const int tx = t % g.px, ty = t / g.px;
    const float* src = in + (int64_t)t * g.tile;
    float* dst = out + (int64_t)t * g.tile;
    const bool active = q < nq;
    const int c = kCol0 + 4 * q;
    const int lane = threadIdx.x & 31;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 up = active ? ld4(src + (int64_t)(r0 - 1) * g.pitch + c) : zero;
    float4 cur = active ? ld4(src + (int64_t)r0 * g.pitch + c) : zero;
    // not unrolled: keeps both variants at 32 registers (full occupancy)
#pragma unroll 1
    for (int r = r0; r < r1; r++) {  // uniform across the block: shuffles see every lane
        const float* row = src + (int64_t)r * g.pitch;
        const float4 dn = active ? ld4(row + g.pitch + c) : zero;
        float w = __shfl_up_sync(kFull, cur.w, 1);
        float e = __shfl_down_sync(kFull, cur.x, 1);
        if (active && lane == 0) w = __ldg(row + c - 1);
        if (active && (lane == 31 || q == nq - 1)) e = __ldg(row + c + 4);
        float4 o;
        o.x = jacobi(up.x, dn.x, w, cur.y);
        o.y = jacobi(up.y, dn.y, cur.x, cur.z);
        o.z = jacobi(up.z, dn.z, cur.y, cur.w);
        o.w = jacobi(up.w, dn.w, cur.z, e);
        if (active) {
            st4(dst + (int64_t)r * g.pitch + c, o);
            if (FUSED) {
                if (r == 1 && ty > 0)
                    st4(out + (int64_t)(t - g.px) * g.tile + (int64_t)(g.n + 1) * g.pitch + c, o);
                if (r == g.n && ty < g.py - 1) st4(out + (int64_t)(t + g.px) * g.tile + c, o);
                if (q == 0 && tx > 0)
                    out[(int64_t)(t - 1) * g.tile + (int64_t)r * g.pitch + kCol0 + g.n] = o.x;
                if (q == nq - 1 && tx < g.px - 1)
                    out[(int64_t)(t + 1) * g.tile + (int64_t)r * g.pitch + kCol0 - 1] = o.w;
            }
        }
        up = cur;
        cur = dn;
    }
}

Geo geo(const stencil_plan* p) { return Geo{p->px, p->py, p->n, p->pitch, p->tile_floats}; }

bool aligned16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }

int launch_sweep(const stencil_plan* p, const float* in, float* out, void* stream, bool fused) {
    if (!p || !aligned16(in) || !aligned16(out) || in == out) return HALO_EINVAL;
    const int nq = p->n / 4;
    const dim3 grid((unsigned)((nq + kQuads - 1) / kQuads), (unsigned)((p->n + kBand - 1) / kBand),
                    (unsigned)(p->px * p->py));
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (fused)
        stencil_sweep_kernel<true><<<grid, kQuads, 0, st>>>(in, out, geo(p));
    else
        stencil_sweep_kernel<false><<<grid, kQuads, 0, st>>>(in, out, geo(p));
    return cudaGetLastError() == cudaSuccess ? HALO_OK : HALO_ECUDA;
}

}  // namespace

extern "C" {

int stencil_setup(int32_t px, int32_t py, int32_t n, stencil_plan** out_plan) {
    if (!out_plan) return HALO_EINVAL;
    *out_plan = nullptr;
    // grid z of the sweep holds the tile index; grid y the row bands
    if (px < 1 || py < 1 || (int64_t)px * py > 65535) return HALO_EINVAL;
    if (n < 4 || n % 4 != 0 || n > (1 << 20)) return HALO_EINVAL;
    stencil_plan* p = new (std::nothrow) stencil_plan();
    if (!p) return HALO_ENOMEM;
    p->px = px;
    p->py = py;
    p->n = n;
    p->pitch = n + 8;
    p->rows = n + 2;
    p->tile_floats = (int64_t)p->rows * p->pitch;
    p->total_floats = p->tile_floats * px * py;
    *out_plan = p;
    return HALO_OK;
}

int stencil_layout(const stencil_plan* p, int32_t* pitch, int32_t* rows, int32_t* col0,
                   int64_t* tile_floats, int64_t* total_floats) {
    if (!p) return HALO_EINVAL;
    if (pitch) *pitch = p->pitch;
    if (rows) *rows = p->rows;
    if (col0) *col0 = kCol0;
    if (tile_floats) *tile_floats = p->tile_floats;
    if (total_floats) *total_floats = p->total_floats;
    return HALO_OK;
}

int stencil_exchange(const stencil_plan* p, float* field, void* stream) {
    if (!p || !aligned16(field)) return HALO_EINVAL;
    if (p->px * p->py == 1) return HALO_OK;  // no neighbours
    const int64_t threads = (int64_t)p->px * p->py * p->n;
    const unsigned blocks = (unsigned)((threads + kExchThreads - 1) / kExchThreads);
    stencil_exchange_kernel<<<blocks, kExchThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        field, geo(p), threads);
    return cudaGetLastError() == cudaSuccess ? HALO_OK : HALO_ECUDA;
}

int stencil_sweep(const stencil_plan* p, const float* in, float* out, void* stream) {
    return launch_sweep(p, in, out, stream, false);
}

int stencil_sweep_fused(const stencil_plan* p, const float* in, float* out, void* stream) {
    return launch_sweep(p, in, out, stream, true);
}

void stencil_destroy(stencil_plan* p) { delete p; }

}  // extern "C"
