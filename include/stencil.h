/*
 * stencil.h -- C ABI of the two-dimensional stencil halo workload in libhalo.so.
 *
 * The second workload of the halo exchange, from the page "GPU-centric
 * Communication on NVIDIA GPU Clusters with InfiniBand: A Case Study with
 * OpenSHMEM", section "2D stencil mini-app": a square matrix split into
 * px x py square blocks (the page's ranks, one- or two-dimensional grid, not
 * periodic); every iteration each block is swept with the stencil and its edge
 * rows and columns go to its up to four neighbours, whose next sweep reads
 * them.  The page compares an MPI version (separate compute and pack kernels,
 * CPU-driven transfers) with a single fused kernel that computes and sends.
 * Here every block lives in one GPU's memory: sending is a store into the
 * neighbour block's ghost cells.
 *
 * Readings where the page is silent: the stencil is the five-point Jacobi
 * sweep, out = ((N + S) + (W + E)) * 0.25 in fp32 (one rounding per operation,
 * in this order); the ghost cells on the matrix border hold fixed values set
 * by the caller that no call writes; only edge rows and columns are exchanged
 * (the five-point stencil reads no diagonal neighbour).
 *
 * Layout of a field (n_tiles = px * py tiles, one after another; tile
 * t = tx + px * ty, tx along the columns, ty along the rows): each tile is
 * n + 2 rows of pitch = n + 8 floats.  Row 0 is the ghost row above the block,
 * rows 1..n the block, row n + 1 the ghost row below; in a row, columns
 * 4 .. n + 3 are the block, column 3 the west ghost, column n + 4 the east
 * ghost, the rest padding (never read or written).  n must be a multiple of 4,
 * so every block row starts 16-byte aligned.
 *
 * All pointers are device pointers to caller-owned fields of
 * stencil_layout()'s total_floats floats, 16-byte aligned.  Calls are
 * asynchronous on `stream` (a cudaStream_t passed as void*, NULL = legacy
 * default stream) and return the HALO_* codes of halo.h: HALO_EINVAL for bad
 * sizes, null or misaligned pointers, or in == out; HALO_ECUDA for a failed
 * launch.
 */
#ifndef STENCIL_H
#define STENCIL_H

#include <stdint.h>

#include "halo.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct stencil_plan stencil_plan; /* opaque; host-side sizes only */

/* A plan for px x py blocks of n x n cells (px, py >= 1; n >= 4, n % 4 == 0).
 * Allocates no device memory (stencil_iterate allocates one small word on
 * first use). */
int stencil_setup(int32_t px, int32_t py, int32_t n, stencil_plan** out_plan);

/* The field layout (host outputs, any may be NULL): floats per row, rows per
 * tile, first block column, floats per tile, floats of the whole field. */
int stencil_layout(const stencil_plan* plan, int32_t* pitch, int32_t* rows, int32_t* col0,
                   int64_t* tile_floats, int64_t* total_floats);

/* Halo exchange of `field`: every block's first row goes to the ghost row
 * below the block above it, its last row to the ghost row above the block
 * below it, its first column to the east ghost column of the block on its
 * left, its last column to the west ghost column of the block on its right.
 * Ghost cells on the matrix border, ghost corners and padding are untouched.
 * One kernel launch. */
int stencil_exchange(const stencil_plan* plan, float* field, void* stream);

/* One Jacobi sweep: every block of `out` from the block and ghost cells of
 * `in`; nothing else of `out` is written.  One kernel launch. */
int stencil_sweep(const stencil_plan* plan, const float* in, float* out, void* stream);

/* The fused iteration (the page's single kernel that computes and sends): the
 * sweep of stencil_sweep, and each new edge value also stored into the
 * neighbouring block's ghost cell of `out`, so that `out` is ready for the
 * next sweep without a separate exchange.  Same result as stencil_sweep
 * followed by stencil_exchange on `out`.  One kernel launch. */
int stencil_sweep_fused(const stencil_plan* plan, const float* in, float* out, void* stream);

/* `iterations` fused iterations in ONE kernel launch, with no host in the
 * loop (the page's GPU-initiated scheme taken to the whole run): iteration i
 * sweeps a into b when i is even, b into a when i is odd, and stores the new
 * edges into the neighbours' ghost cells; the blocks of the launch meet at a
 * grid-wide barrier between iterations.  The result is in a when iterations
 * is even, in b when it is odd; a and b must hold the same matrix border and
 * a must hold valid ghost cells (after stencil_exchange or a fused step).
 * Same result as that many stencil_sweep_fused calls.  The launch is
 * cooperative (all its blocks resident at once); every barrier wait is
 * bounded (1 s): a wait that runs out records HALO_ETIMEOUT for
 * stencil_status and the kernel returns.  The first call allocates the
 * barrier's 64-byte device word for the plan.  iterations >= 0. */
int stencil_iterate(stencil_plan* plan, float* a, float* b, int32_t iterations, void* stream);

/* Synchronise `stream` and return (and clear) the error recorded by the last
 * stencil_iterate: HALO_OK or HALO_ETIMEOUT. */
int stencil_status(stencil_plan* plan, void* stream);

void stencil_destroy(stencil_plan* plan);

#ifdef __cplusplus
}
#endif

#endif /* STENCIL_H */
