// halo_api.cu -- the C ABI of libhalo.so (declared in include/halo.h).
//
// Argument checks, plan ownership and the pulse bookkeeping of the page
// "Redesigning GROMACS Halo Exchange: Improving Strong Scaling with
// GPU-initiated NVSHMEM" (review): section 3 (np(z) pulses in z, then np(y) in
// y, then np(x) in x) and section 4 (Total Pulses = np(x)+np(y)+np(z)); the
// device work lives in halo_build.cu and halo_exchange.cu.
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <new>

#include "halo_internal.cuh"

namespace {

// Make the plan's device current for the duration of a call.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            ok = false;
            prev = -1;
            return;
        }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

int check_problem(const float box[3], const int32_t grid[3], float rc, halo_plan* pl) {
    if (!box || !grid) return HALO_EINVAL;
    if (!(rc > 0.0f) || !isfinite(rc)) return HALO_EINVAL;
    int64_t nd = 1;
    for (int d = 0; d < 3; d++) {
        if (grid[d] < 1 || !(box[d] > 0.0f) || !isfinite(box[d])) return HALO_EINVAL;
        nd *= grid[d];
    }
    if (nd > HALO_MAX_DOMAINS) return HALO_EINVAL;
    int P = 0;
    int per[3] = {0, 0, 0};
    for (int d = 0; d < 3; d++) {
        if (grid[d] > 1) {
            const double w = (double)box[d] / (double)grid[d];
            const double pc = ceil((double)rc / w);
            if (pc >= (double)grid[d]) return HALO_EPULSES;
            per[d] = (int)pc;
        }
        P += per[d];
    }
    if (P > HALO_MAX_PULSES) return HALO_EINVAL;
    if (pl) {
        for (int d = 0; d < 3; d++) {
            pl->grid[d] = grid[d];
            pl->box[d] = box[d];
            pl->pulses_per_dim[d] = per[d];
        }
        pl->rc = rc;
        pl->n_dom = (int)nd;
        pl->P = 0;
        for (int d = 2; d >= 0; d--)
            for (int k = 0; k < per[d]; k++) {
                pl->pulse_dim[pl->P] = d;
                pl->pulse_k[pl->P] = k;
                pl->P++;
            }
    }
    return HALO_OK;
}

void destroy_plan(halo_plan* pl) {
    if (!pl) return;
    {
        DeviceGuard g(pl->dev);
        halo::free_exchange(pl);
        halo::free_flat(pl);
        halo::free_build(pl);
        if (pl->h_stage) cudaFreeHost(pl->h_stage);
        pl->h_stage = nullptr;
        pl->h_stage_dev = nullptr;
    }
    delete pl;
}

int do_build(halo_plan* pl, const float* coords, const int32_t* dom, int64_t n, void* stream) {
    const cudaStream_t st = as_stream(stream);
    pl->valid = false;  // until every table of the new plan is in place
    pl->trace = nullptr;  // item counts change with the plan: the caller re-arms tracing
    pl->trace_cap = 0;
    pl->flat_ready = false;  // the flattened tables describe the previous plan
    pl->flat_chains_ready = false;
    HALO_TRY(halo::build_plan(pl, coords, dom, n, st));
    // FLAT: the forwarding chains need only the device's descriptors and the
    // sizes, so the GPU runs them while the host builds its copy of the
    // descriptors below
    if (pl->mode == HALO_MODE_FLAT) HALO_TRY(halo::launch_flat_chains(pl, st));
    halo::update_shard_first(pl);
    HALO_TRY(halo::prepare_common(pl, st));
    // each mode's own tables; the others are built when a mode is selected
    // (the sharded data plane runs on the FUSED work lists)
    if (pl->mode == HALO_MODE_FUSED || pl->shard_lists) HALO_TRY(halo::prepare_fused(pl, st));
    if (pl->mode == HALO_MODE_FLAT) HALO_TRY(halo::prepare_flat(pl, st));
    if (pl->mode == HALO_MODE_STAGED) HALO_TRY(halo::prepare_staged(pl));
    pl->valid = true;
    return HALO_OK;
}

}  // namespace

extern "C" {

int halo_setup(const float box[3], const int32_t grid[3], float rc, const float* coords,
               const int32_t* domain_of_atom, int64_t n_atoms, void* stream,
               halo_plan** out_plan) {
    return halo_setup_ex(box, grid, rc, coords, domain_of_atom, n_atoms, 0u, stream, out_plan);
}

int halo_setup_ex(const float box[3], const int32_t grid[3], float rc, const float* coords,
                  const int32_t* domain_of_atom, int64_t n_atoms, uint32_t flags, void* stream,
                  halo_plan** out_plan) {
    if (!out_plan) return HALO_EINVAL;
    *out_plan = nullptr;
    if (!coords || !domain_of_atom || n_atoms <= 0 || n_atoms > INT32_MAX / 2)
        return HALO_EINVAL;
    if (flags & ~HALO_SETUP_PRUNE_CORNERS) return HALO_EINVAL;
    HALO_TRY(check_problem(box, grid, rc, nullptr));
    halo_plan* pl = new (std::nothrow) halo_plan();
    if (!pl) return HALO_ENOMEM;
    int rc_ = HALO_OK;
    pl->flags = flags;
    if (const char* env = getenv("HALO_WAIT_TIMEOUT_MS")) {
        const double ms = atof(env);
        if (ms > 0.0 && isfinite(ms)) pl->wait_timeout_ns = (long long)(ms * 1e6);
    }
    if (const char* env = getenv("HALO_STAGE_COPIES")) pl->stage_copies = env[0] != '\0' && strcmp(env, "0") != 0;
    try {
        rc_ = check_problem(box, grid, rc, pl);
        if (rc_ == HALO_OK && cudaGetDevice(&pl->dev) != cudaSuccess) rc_ = HALO_ECUDA;
        if (rc_ == HALO_OK &&
            cudaDeviceGetAttribute(&pl->num_sms, cudaDevAttrMultiProcessorCount, pl->dev) !=
                cudaSuccess)
            rc_ = HALO_ECUDA;
        // the fixed array of halo_exchange_x_noalloc gets its device address
        // here, so that call never loads or places anything itself
        if (rc_ == HALO_OK) rc_ = halo::noalloc_prepare();
        if (rc_ == HALO_OK) rc_ = halo::set_shards(pl, 1);  // one shard: the dense buffer
        if (rc_ == HALO_OK) rc_ = do_build(pl, coords, domain_of_atom, n_atoms, stream);
    } catch (const std::bad_alloc&) {
        rc_ = HALO_ENOMEM;
    } catch (...) {
        rc_ = HALO_ECUDA;
    }
    if (rc_ != HALO_OK) {
        destroy_plan(pl);
        return rc_;
    }
    *out_plan = pl;
    return HALO_OK;
}

int halo_rebuild(halo_plan* pl, const float* coords, const int32_t* domain_of_atom,
                 int64_t n_atoms, void* stream) {
    if (!pl || !coords || !domain_of_atom || n_atoms <= 0 || n_atoms > INT32_MAX / 2)
        return HALO_EINVAL;
    DeviceGuard g(pl->dev);
    if (!g.ok) return HALO_ECUDA;
    try {
        return do_build(pl, coords, domain_of_atom, n_atoms, stream);
    } catch (const std::bad_alloc&) {
        return HALO_ENOMEM;
    } catch (...) {
        return HALO_ECUDA;
    }
}

int halo_query(const halo_plan* pl, halo_info* out) {
    if (!pl || !out) return HALO_EINVAL;
    memset(out, 0, sizeof(*out));
    out->n_domains = pl->n_dom;
    out->n_pulses = pl->P;
    for (int d = 0; d < 3; d++) out->pulses_per_dim[d] = pl->pulses_per_dim[d];
    for (int p = 0; p < pl->P; p++) out->pulse_dim[p] = pl->pulse_dim[p];
    out->flags = pl->flags;
    out->build_attempts = pl->build_attempts;
    out->n_atoms = pl->n_atoms;
    out->n_local_total = pl->n_local_total;
    out->n_halo_total = pl->n_halo_total;
    return HALO_OK;
}

int halo_domain_layout(const halo_plan* pl, int64_t* base, int32_t* n_home, int32_t* n_local) {
    if (!pl || !pl->valid) return HALO_EINVAL;
    for (int D = 0; D < pl->n_dom; D++) {
        if (base) base[D] = pl->base[D];
        if (n_home) n_home[D] = pl->n_home[D];
        if (n_local) n_local[D] = pl->n_local[D];
    }
    return HALO_OK;
}

int halo_get_pulse(const halo_plan* pl, int32_t domain, int32_t pulse, halo_pulse_info* out,
                   int32_t* index_map) {
    if (!pl || !out || !pl->valid || domain < 0 || domain >= pl->n_dom || pulse < 0 ||
        pulse >= pl->P)
        return HALO_EINVAL;
    const halo::SPDesc& d = pl->sp[(size_t)domain * pl->P + pulse];
    out->send_domain = domain;
    out->recv_domain = d.r;
    out->send_size = d.send;
    out->split = d.split;
    out->dep_offset = pl->n_home[domain];
    out->atom_offset = pl->own_off[(size_t)d.r * (pl->P + 1) + pulse];
    for (int e = 0; e < 3; e++) out->coord_shift[e] = d.shift[e];
    if (index_map && d.send > 0) {
        DeviceGuard g(pl->dev);
        if (!g.ok) return HALO_ECUDA;
        HALO_CUDA(cudaMemcpy(index_map, pl->d_maps + d.map_off, sizeof(int32_t) * d.send,
                             cudaMemcpyDeviceToHost));
    }
    return HALO_OK;
}

int halo_get_index_maps(const halo_plan* pl, int32_t* maps, int64_t* offsets) {
    if (!pl || !offsets || !pl->valid || (!maps && pl->n_halo_total > 0)) return HALO_EINVAL;
    const int nd = pl->n_dom, P = pl->P;
    for (int p = 0; p < P; p++)
        for (int s = 0; s < nd; s++) offsets[(size_t)p * nd + s] = pl->map_off[(size_t)s * P + p];
    offsets[(size_t)P * nd] = pl->n_halo_total;
    if (pl->n_halo_total > 0) {
        DeviceGuard g(pl->dev);
        if (!g.ok) return HALO_ECUDA;
        HALO_CUDA(cudaMemcpy(maps, pl->d_maps, sizeof(int32_t) * (size_t)pl->n_halo_total,
                             cudaMemcpyDeviceToHost));
    }
    return HALO_OK;
}

int halo_local_to_global(const halo_plan* pl, int32_t* out, void* stream) {
    if (!pl || !out || !pl->valid) return HALO_EINVAL;
    DeviceGuard g(pl->dev);
    if (!g.ok) return HALO_ECUDA;
    return halo::launch_local_to_global(pl, out, as_stream(stream));
}

int halo_load_home(const halo_plan* pl, const float* global_xyz, float* local_xyz, void* stream) {
    if (!pl || !global_xyz || !local_xyz || !pl->valid) return HALO_EINVAL;
    DeviceGuard g(pl->dev);
    if (!g.ok) return HALO_ECUDA;
    return halo::launch_load_home(pl, global_xyz, local_xyz, as_stream(stream));
}

int halo_store_home(const halo_plan* pl, const float* local_xyz, float* global_xyz, void* stream) {
    if (!pl || !global_xyz || !local_xyz || !pl->valid) return HALO_EINVAL;
    DeviceGuard g(pl->dev);
    if (!g.ok) return HALO_ECUDA;
    return halo::launch_store_home(pl, local_xyz, global_xyz, as_stream(stream));
}

int halo_exchange_x(halo_plan* pl, float* local_coords, void* stream) {
    if (!pl || !local_coords || ((uintptr_t)local_coords & 3u)) return HALO_EINVAL;
    if (!pl->valid) return HALO_EINVAL;
    DeviceGuard g(pl->dev);
    if (!g.ok) return HALO_ECUDA;
    switch (pl->mode) {
        case HALO_MODE_STEPWISE: return halo::launch_stepwise_x(pl, local_coords, as_stream(stream));
        case HALO_MODE_FLAT: return halo::launch_flat_x(pl, local_coords, as_stream(stream));
        case HALO_MODE_STAGED: return halo::launch_staged_x(pl, local_coords, as_stream(stream));
        default: return halo::launch_exchange_x(pl, local_coords, as_stream(stream));
    }
}

int halo_exchange_f(halo_plan* pl, float* local_forces, void* stream) {
    if (!pl || !local_forces || ((uintptr_t)local_forces & 3u)) return HALO_EINVAL;
    if (!pl->valid) return HALO_EINVAL;
    DeviceGuard g(pl->dev);
    if (!g.ok) return HALO_ECUDA;
    switch (pl->mode) {
        case HALO_MODE_STEPWISE: return halo::launch_stepwise_f(pl, local_forces, as_stream(stream));
        case HALO_MODE_FLAT: return halo::launch_flat_f(pl, local_forces, as_stream(stream));
        case HALO_MODE_STAGED: return halo::launch_staged_f(pl, local_forces, as_stream(stream));
        default: return halo::launch_exchange_f(pl, local_forces, as_stream(stream));
    }
}

// ---- sharded data plane -------------------------------------------------------

int halo_shard(halo_plan* pl, int32_t n_shards, void* stream) {
    if (!pl || !pl->valid) return HALO_EINVAL;
    DeviceGuard g(pl->dev);
    if (!g.ok) return HALO_ECUDA;
    HALO_TRY(halo::set_shards(pl, n_shards));
    pl->shard_lists = true;
    // the work lists carry each item's shards
    return halo::prepare_fused(pl, as_stream(stream));
}

int halo_shard_layout(const halo_plan* pl, int32_t shard, int32_t* first_domain, int32_t* n_domains,
                      int64_t* first_slot, int64_t* n_local) {
    if (!pl || !pl->valid || shard < 0 || shard >= pl->n_shards) return HALO_EINVAL;
    if (first_domain) *first_domain = pl->shard_dom[shard];
    if (n_domains) *n_domains = pl->shard_dom[shard + 1] - pl->shard_dom[shard];
    if (first_slot) *first_slot = pl->shard_first[shard];
    if (n_local) *n_local = pl->shard_first[shard + 1] - pl->shard_first[shard];
    return HALO_OK;
}

namespace {
bool shard_ptrs_ok(const halo_plan* pl, const void* const* p) {
    if (!p) return false;
    for (int k = 0; k < pl->n_shards; k++)
        if (!p[k] || ((uintptr_t)p[k] & 3u)) return false;
    return true;
}
}  // namespace

int halo_load_home_sharded(const halo_plan* pl, const float* global_xyz, float* const* shard_local,
                           void* stream) {
    if (!pl || !global_xyz || !pl->valid || !shard_ptrs_ok(pl, (const void* const*)shard_local))
        return HALO_EINVAL;
    DeviceGuard g(pl->dev);
    if (!g.ok) return HALO_ECUDA;
    return halo::launch_load_home_sharded(pl, global_xyz, shard_local, as_stream(stream));
}

int halo_store_home_sharded(const halo_plan* pl, const float* const* shard_local, float* global_xyz,
                            void* stream) {
    if (!pl || !global_xyz || !pl->valid || !shard_ptrs_ok(pl, (const void* const*)shard_local))
        return HALO_EINVAL;
    DeviceGuard g(pl->dev);
    if (!g.ok) return HALO_ECUDA;
    return halo::launch_store_home_sharded(pl, shard_local, global_xyz, as_stream(stream));
}

int halo_exchange_x_sharded(halo_plan* pl, float* const* shard_coords, void* stream) {
    if (!pl || !pl->valid || !pl->fused_ready || !shard_ptrs_ok(pl, (const void* const*)shard_coords))
        return HALO_EINVAL;
    DeviceGuard g(pl->dev);
    if (!g.ok) return HALO_ECUDA;
    return halo::launch_exchange_x_sharded(pl, shard_coords, as_stream(stream));
}

int halo_exchange_f_sharded(halo_plan* pl, float* const* shard_forces, void* stream) {
    if (!pl || !pl->valid || !pl->fused_ready || !shard_ptrs_ok(pl, (const void* const*)shard_forces))
        return HALO_EINVAL;
    DeviceGuard g(pl->dev);
    if (!g.ok) return HALO_ECUDA;
    return halo::launch_exchange_f_sharded(pl, shard_forces, as_stream(stream));
}

int halo_status(halo_plan* pl, void* stream) {
    if (!pl) return HALO_EINVAL;
    DeviceGuard g(pl->dev);
    if (!g.ok) return HALO_ECUDA;
    const cudaStream_t st = as_stream(stream);
    HALO_CUDA(cudaStreamSynchronize(st));
    HALO_CUDA(cudaGetLastError());
    int e[8] = {0};
    if (pl->d_err) HALO_CUDA(cudaMemcpy(e, pl->d_err, sizeof(e), cudaMemcpyDeviceToHost));
    if (e[0] != HALO_OK) {
        HALO_TRY(halo::reset_flags(pl, st));
        HALO_CUDA(cudaStreamSynchronize(st));
    }
    return e[0];
}

int halo_debug_set_build_capacity(halo_plan* pl, int64_t slots) {
    if (!pl || slots <= 0) return HALO_EINVAL;
    pl->debug_capacity = slots;
    return HALO_OK;
}

int halo_set_wait_timeout(halo_plan* pl, double seconds) {
    if (!pl || !(seconds > 0.0) || !isfinite(seconds)) return HALO_EINVAL;
    pl->wait_timeout_ns = (long long)(seconds * 1e9);
    return HALO_OK;
}

int halo_debug_drop_signal(halo_plan* pl, int32_t domain, int32_t pulse) {
    if (!pl) return HALO_EINVAL;
    if (domain == -1 && pulse == -1) {
        pl->drop_flag = -1;
        return HALO_OK;
    }
    if (domain < 0 || domain >= pl->n_dom || pulse < 0 || pulse >= pl->P) return HALO_EINVAL;
    // the counter the producer (domain, pulse) releases: arrived[r*P + pulse]
    pl->drop_flag = pl->sp[(size_t)domain * pl->P + pulse].r * pl->P + pulse;
    return HALO_OK;
}

int halo_set_mode(halo_plan* pl, int32_t mode, void* stream) {
    if (!pl) return HALO_EINVAL;
    if (mode != HALO_MODE_FUSED && mode != HALO_MODE_STEPWISE && mode != HALO_MODE_FLAT &&
        mode != HALO_MODE_STAGED)
        return HALO_EINVAL;
    DeviceGuard g(pl->dev);
    if (!g.ok) return HALO_ECUDA;
    const bool build = (mode == HALO_MODE_FUSED && !pl->fused_ready) ||
                       (mode == HALO_MODE_FLAT && !pl->flat_ready) || mode == HALO_MODE_STAGED;
    if (build && !pl->valid) return HALO_EINVAL;  // a failed rebuild: nothing to build from
    try {
        if (mode == HALO_MODE_FUSED && !pl->fused_ready) HALO_TRY(halo::prepare_fused(pl, as_stream(stream)));
        if (mode == HALO_MODE_FLAT && !pl->flat_ready) HALO_TRY(halo::prepare_flat(pl, as_stream(stream)));
        if (mode == HALO_MODE_STAGED) HALO_TRY(halo::prepare_staged(pl));
    } catch (const std::bad_alloc&) {
        return HALO_ENOMEM;
    }
    pl->mode = mode;
    return HALO_OK;
}

int halo_get_mode(const halo_plan* pl, int32_t* mode) {
    if (!pl || !mode) return HALO_EINVAL;
    *mode = pl->mode;
    return HALO_OK;
}

int halo_set_trace(halo_plan* pl, uint64_t* trace, int64_t capacity_items) {
    if (!pl) return HALO_EINVAL;
    if (!trace) {
        pl->trace = nullptr;
        pl->trace_cap = 0;
        return HALO_OK;
    }
    if (!pl->fused_ready || capacity_items < (int64_t)pl->n_items_x + pl->n_items_f) return HALO_EINVAL;
    pl->trace = reinterpret_cast<unsigned long long*>(trace);
    pl->trace_cap = capacity_items;
    return HALO_OK;
}

int halo_work_items(const halo_plan* pl, int32_t* x_items, int32_t* f_items, int32_t* chunk) {
    if (!pl || !pl->fused_ready) return HALO_EINVAL;
    if (x_items) *x_items = pl->n_items_x;
    if (f_items) *f_items = pl->n_items_f;
    if (chunk) *chunk = pl->chunk;
    return HALO_OK;
}

int halo_launch_counts(const halo_plan* pl, int64_t* x_launches, int64_t* f_launches) {
    if (!pl) return HALO_EINVAL;
    if (x_launches) *x_launches = pl->launches_x;
    if (f_launches) *f_launches = pl->launches_f;
    return HALO_OK;
}

void halo_destroy(halo_plan* pl) { destroy_plan(pl); }

const char* halo_strerror(int code) {
    switch (code) {
        case HALO_OK: return "ok";
        case HALO_EINVAL: return "invalid argument";
        case HALO_EPULSES: return "cut-off needs as many pulses as domains in a dimension";
        case HALO_EDOMAIN: return "domain id out of range";
        case HALO_ECAPACITY: return "build buffer capacity exhausted";
        case HALO_ECUDA: return "CUDA runtime error";
        case HALO_ETIMEOUT: return "device-side wait timed out";
        case HALO_EBOUNDS: return "index out of bounds";
        case HALO_ENOMEM: return "out of memory";
        case HALO_ESCRATCH: return "plan too large for the fixed scratch of halo_exchange_x_noalloc";
        default: return "unknown error";
    }
}

}  // extern "C"
