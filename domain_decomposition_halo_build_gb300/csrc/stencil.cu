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

#include <algorithm>
#include <new>

#include "stencil.h"

struct stencil_plan {
    int px = 0, py = 0, n = 0;
    int pitch = 0, rows = 0;
    int64_t tile_floats = 0, total_floats = 0;
    // stencil_iterate: barrier counter and error word (allocated on first use)
    unsigned* d_sync = nullptr;
    int dev = -1;
    int iterate_grid = 0;  // co-resident blocks of the persistent kernel
    int band = 16;         // rows per sweep unit
};

namespace {

constexpr int kCol0 = 4;     // first block column of a tile row
constexpr int kQuads = 128;  // threads per sweep block, 4 cells each
constexpr int kBand = 16;    // rows per sweep unit (at most; fewer for small blocks)
constexpr int kMinUnits = 1024;  // sweep units wanted per launch before bands shrink
constexpr int kExchThreads = 256;
constexpr unsigned kFull = 0xffffffffu;

struct Geo {
    int px, py, n, pitch;
    int64_t tile;  // floats per tile
    int band;      // rows per sweep unit
};

__device__ __forceinline__ float4 ld4(const float* p) {
    return __ldg(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }

// loads of a sweep's input: non-coherent path, or L2 when the input was
// written earlier in the same launch
template <bool COHERENT>
__device__ __forceinline__ float4 ld4c(const float* p) {
    return COHERENT ? __ldcg(reinterpret_cast<const float4*>(p)) : ld4(p);
}
template <bool COHERENT>
__device__ __forceinline__ float ld1c(const float* p) {
    return COHERENT ? __ldcg(p) : __ldg(p);
}

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

// One unit of a sweep: 512 columns (128 threads x 4) of block t over the
// band of rows starting at 1 + by * g.band.  COHERENT: `in` was written earlier
// in the same launch (the persistent kernel), so it is read through L2 (.cg)
// rather than the non-coherent path.
template <bool FUSED, bool COHERENT>
__device__ __forceinline__ void sweep_unit(const float* __restrict__ in, float* out, const Geo& g,
                                           int cx, int by, int t) {
    const int nq = g.n / 4;
    const int q = cx * kQuads + threadIdx.x;  // group of 4 columns
    const int r0 = 1 + by * g.band;            // first row of the band (<= n)
    const int r1 = min(r0 + g.band, g.n + 1);  // one past its last row
    const int tx = t % g.px, ty = t / g.px;
    const float* src = in + (int64_t)t * g.tile;
    float* dst = out + (int64_t)t * g.tile;
    const bool active = q < nq;
    const int c = kCol0 + 4 * q;
    const int lane = threadIdx.x & 31;
    const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 up = active ? ld4c<COHERENT>(src + (int64_t)(r0 - 1) * g.pitch + c) : zero;
    float4 cur = active ? ld4c<COHERENT>(src + (int64_t)r0 * g.pitch + c) : zero;
    // not unrolled: keeps both variants at 32 registers (full occupancy)
#pragma unroll 1
    for (int r = r0; r < r1; r++) {  // uniform across the block: shuffles see every lane
        const float* row = src + (int64_t)r * g.pitch;
        const float4 dn = active ? ld4c<COHERENT>(row + g.pitch + c) : zero;
        float w = __shfl_up_sync(kFull, cur.w, 1);
        float e = __shfl_down_sync(kFull, cur.x, 1);
        if (active && lane == 0) w = ld1c<COHERENT>(row + c - 1);
        if (active && (lane == 31 || q == nq - 1)) e = ld1c<COHERENT>(row + c + 4);
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

template <bool FUSED>
__global__ void __launch_bounds__(kQuads) stencil_sweep_kernel(const float* __restrict__ in,
                                                               float* out, Geo g) {
    sweep_unit<FUSED, false>(in, out, g, blockIdx.x, blockIdx.y, blockIdx.z);
}

__device__ __forceinline__ unsigned ld_acquire_gpu_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Grid-wide barrier of a cooperative launch: every block arrives once per
// iteration on a counter that only grows, then waits until all gridDim.x
// blocks of this iteration have arrived.  The wait is bounded: past
// timeout_ns it records HALO_ETIMEOUT and gives up (as does every other block
// once it sees the error), and the kernel returns.
__device__ __forceinline__ bool grid_barrier(unsigned* count, int* err, unsigned target,
                                             long long timeout_ns) {
    __shared__ int s_ok;
    __syncthreads();  // this block's stores of the iteration are issued
    if (threadIdx.x == 0) {
        __threadfence();  // ... and visible to the whole GPU before arriving
        atomicAdd(count, 1u);
        int ok = 1;
        const uint64_t t0 = global_timer_ns();
        unsigned ns = 32;
        while (ld_acquire_gpu_u32(count) < target) {
            if (*(volatile int*)err != 0) {
                ok = 0;
                break;
            }
            if ((long long)(global_timer_ns() - t0) > timeout_ns) {
                atomicCAS(err, 0, HALO_ETIMEOUT);
                ok = 0;
                break;
            }
            __nanosleep(ns);
            if (ns < 256) ns *= 2;
        }
        __threadfence();
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// `iters` fused iterations in one cooperative launch: a -> b, b -> a, ...;
// the blocks share the sweep units of an iteration (grid-stride) and meet at
// the barrier before the next one reads what this one wrote.
__global__ void __launch_bounds__(kQuads) stencil_iterate_kernel(float* a, float* b, Geo g, int iters,
                                                                 int units_x, int units_y,
                                                                 unsigned* count, int* err,
                                                                 long long timeout_ns) {
    const int64_t per_tile = (int64_t)units_x * units_y;
    const int64_t units = per_tile * g.px * g.py;
    for (int it = 0; it < iters; it++) {
        const float* in = (it & 1) ? b : a;
        float* out = (it & 1) ? a : b;
        for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
            const int t = (int)(u / per_tile);
            const int64_t v = u - (int64_t)t * per_tile;
            sweep_unit<true, true>(in, out, g, (int)(v % units_x), (int)(v / units_x), t);
        }
        if (it + 1 < iters && !grid_barrier(count, err, (unsigned)(it + 1) * gridDim.x, timeout_ns))
            return;
    }
}

Geo geo(const stencil_plan* p) { return Geo{p->px, p->py, p->n, p->pitch, p->tile_floats, p->band}; }

bool aligned16(const void* p) { return p && ((uintptr_t)p & 15u) == 0; }

int launch_sweep(const stencil_plan* p, const float* in, float* out, void* stream, bool fused) {
    if (!p || !aligned16(in) || !aligned16(out) || in == out) return HALO_EINVAL;
    const int nq = p->n / 4;
    const dim3 grid((unsigned)((nq + kQuads - 1) / kQuads), (unsigned)((p->n + p->band - 1) / p->band),
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
    // rows per sweep unit: 16 (each input row read once per 16 output rows,
    // plus the two around them) unless that leaves too few units to keep the
    // GPU's warps busy, when the per-thread chain of row loads is the limit;
    // then 8 or 4
    const int64_t cols = ((int64_t)n / 4 + kQuads - 1) / kQuads;
    p->band = kBand;
    while (p->band > 4 && cols * ((n + p->band - 1) / p->band) * px * py < kMinUnits) p->band /= 2;
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

int stencil_iterate(stencil_plan* p, float* a, float* b, int32_t iterations, void* stream) {
    if (!p || !aligned16(a) || !aligned16(b) || a == b || iterations < 0) return HALO_EINVAL;
    if (iterations == 0) return HALO_OK;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return HALO_ECUDA;
    if (!p->d_sync || p->dev != dev) {
        if (p->d_sync) cudaFree(p->d_sync);
        p->d_sync = nullptr;
        if (cudaMalloc(&p->d_sync, 64) != cudaSuccess) return HALO_ENOMEM;
        p->dev = dev;
        int sms = 0, occ = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, stencil_iterate_kernel, kQuads, 0) !=
                cudaSuccess)
            return HALO_ECUDA;
        p->iterate_grid = sms * occ;
    }
    const int units_x = (p->n / 4 + kQuads - 1) / kQuads;
    const int units_y = (p->n + p->band - 1) / p->band;
    const int64_t units = (int64_t)units_x * units_y * p->px * p->py;
    const int grid = (int)std::min<int64_t>(units, p->iterate_grid);
    // the barrier counter reaches iterations * grid
    if ((int64_t)iterations * grid >= ((int64_t)1 << 31)) return HALO_EINVAL;
    if (cudaMemsetAsync(p->d_sync, 0, 64, st) != cudaSuccess) return HALO_ECUDA;
    Geo g = geo(p);
    int iters = iterations;
    int ux = units_x, uy = units_y;
    unsigned* count = p->d_sync;
    int* err = reinterpret_cast<int*>(p->d_sync + 4);
    long long timeout_ns = 1000000000LL;
    void* args[] = {&a, &b, &g, &iters, &ux, &uy, &count, &err, &timeout_ns};
    const cudaError_t e = cudaLaunchCooperativeKernel((const void*)stencil_iterate_kernel, dim3(grid),
                                                      dim3(kQuads), args, 0, st);
    return e == cudaSuccess ? HALO_OK : HALO_ECUDA;
}

int stencil_status(stencil_plan* p, void* stream) {
    if (!p) return HALO_EINVAL;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return HALO_ECUDA;
    if (!p->d_sync) return HALO_OK;
    int e = 0;
    if (cudaMemcpy(&e, p->d_sync + 4, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return HALO_ECUDA;
    if (e != HALO_OK && cudaMemset(p->d_sync + 4, 0, sizeof(int)) != cudaSuccess) return HALO_ECUDA;
    return e;
}

void stencil_destroy(stencil_plan* p) {
    if (p && p->d_sync) cudaFree(p->d_sync);
    delete p;
}

}  // extern "C"
