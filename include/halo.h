/*
 * halo.h -- C ABI of libhalo.so: the eighth-shell domain-decomposition halo
 * exchange of a molecular-dynamics code, with every domain of the periodic box
 * resident in one GPU's memory (GB300, sm_103a).
 *
 * What it computes (page "Redesigning GROMACS Halo Exchange: Improving Strong
 * Scaling with GPU-initiated NVSHMEM", review):
 *   - section 3 "GROMACS domain-decomposition halo exchange": the box is split
 *     into n = (nx, ny, nz) domains, each owning its home atoms; atoms within
 *     the cut-off rc of a domain face are sent to the neighbour and forwarded
 *     through intermediate domains (eighth shell), np(z) pulses in z, then
 *     np(y) in y, then np(x) in x;
 *   - Algorithm 1: per pulse an index map (sendSize entries), the receiver's
 *     atomOffset and a periodic coordShift;
 *   - Algorithms 3/4 (FusedPackCommX, packWithDeps): one launch packs every
 *     pulse; entries below depOffset are independent, the others wait for the
 *     pulse that delivered them;
 *   - Algorithm 6 (FusedCommUnpackF): one launch adds every halo force back to
 *     its owner, pulses from the last to the first.
 *
 * Conventions (fixed by this library where the page is silent):
 *   - domain id D = ix + nx*(iy + ny*iz);
 *   - p_d = ceil(rc / (L_d/n_d)) pulses in each dim with n_d > 1, 0 otherwise;
 *     global pulse order z0..z(pz-1), y0.., x0..; P = pz + py + px <= 64;
 *   - coordinates flow from sender s to receiver r = s - e_d (periodic), so a
 *     domain's halo lies above its upper faces; forces flow back from r to s;
 *   - an atom of s is selected for a pulse of dim d iff x_d < thr, one fp32
 *     compare with thr = fl32(s_d*L_d/n_d + rc) evaluated in double; pulse 0 of
 *     a dim selects among s's home atoms and all halo of earlier dims, pulse
 *     k >= 1 only among the slots s received in pulse k-1 of the same dim;
 *   - index maps are ascending local indices; depOffset = n_home[s]; split =
 *     number of entries < depOffset;
 *   - coordShift = +L_d on component d iff s_d == 0, else 0;
 *   - local layout of domain D: [home atoms in input order | halo of pulse 0 |
 *     ... | halo of pulse P-1]; the dense buffers hold all domains back to
 *     back, domain D starting at slot base[D] = sum of n_local of lower ids;
 *   - coordinates and forces are fp32 AoS xyz (12 bytes per slot).
 *
 * Pointers are DEVICE pointers unless marked (host).  `stream` is a
 * cudaStream_t passed as void* (NULL = legacy default stream).  Exchanges are
 * asynchronous on `stream`; halo_setup / halo_rebuild synchronise `stream` to
 * read the sizes back and return with all the work they queued on it done.
 * A plan is used by one stream at a time.  Every call
 * returns HALO_OK or a negative error code; no exception crosses the ABI.
 * Errors met by a kernel (a bounded wait that gave up) are sticky in the plan
 * and are returned, and cleared, by halo_status().
 */
#ifndef HALO_H
#define HALO_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define HALO_OK 0
#define HALO_EINVAL (-1)    /* null pointer, non-positive L / rc / n, n_atoms <= 0 */
#define HALO_EPULSES (-2)   /* p_d >= n_d: the halo would wrap onto its own domain */
#define HALO_EDOMAIN (-3)   /* a domain id outside [0, nx*ny*nz) */
#define HALO_ECAPACITY (-4) /* build buffers could not be sized (internal retries exhausted) */
#define HALO_ECUDA (-5)     /* a CUDA runtime call failed */
#define HALO_ETIMEOUT (-6)  /* a device-side wait gave up after the plan's time limit */
#define HALO_EBOUNDS (-7)   /* an index outside its buffer was met and skipped (bounds-checking
                               build libhalo_debug.so only) */
#define HALO_ENOMEM (-8)    /* device or host allocation failed */
#define HALO_ESCRATCH (-9)  /* the plan needs more counters than halo_exchange_x_noalloc's fixed array */

/* Exchange modes (halo_set_mode).  All four compute bit-identical results. */
#define HALO_MODE_FUSED 0    /* one launch per direction, per-(domain, pulse) signals (default) */
#define HALO_MODE_STEPWISE 1 /* one launch per pulse and direction, ordered by the stream */
#define HALO_MODE_FLAT 2     /* forwarding chains composed at build time, one wait-free pass */
#define HALO_MODE_STAGED 3   /* MPI-era baseline: pack, host wait, transfer, host wait per pulse */

#define HALO_MAX_PULSES 64
#define HALO_MAX_SHARDS 8
#define HALO_MAX_DOMAINS 4096

typedef struct halo_plan halo_plan; /* opaque; owns maps, metadata, flags, build buffers */

typedef struct {
    int32_t n_domains;
    int32_t n_pulses;
    int32_t pulses_per_dim[3];              /* p_x, p_y, p_z */
    int32_t pulse_dim[HALO_MAX_PULSES];     /* dim (0=x,1=y,2=z) of each global pulse */
    int64_t n_atoms;
    int64_t n_local_total;                  /* home + halo slots of all domains */
    int64_t n_halo_total;
    uint32_t flags;                         /* HALO_SETUP_* flags the plan was built with */
    int32_t build_attempts;                 /* passes the last build needed: 1, or more when the
                                               build buffer overflowed and was grown (retry) */
} halo_info;

typedef struct {
    int32_t send_domain;   /* s */
    int32_t recv_domain;   /* r = s - e_d (periodic) */
    int32_t send_size;     /* index-map entries (= halo slots the receiver gets) */
    int32_t split;         /* entries < dep_offset: independent of earlier pulses */
    int32_t dep_offset;    /* = n_home[s] */
    int32_t atom_offset;   /* first halo slot of this pulse in the receiver's local range */
    float coord_shift[3];  /* added to every packed coordinate */
} halo_pulse_info;

/* Build a plan: pulses, home partition and every pulse's index map, on the
 * device (Algorithm 1's PulseData for all domains).
 *   box (host, 3 floats, nm), grid (host, 3 ints), rc (nm);
 *   coords: n_atoms x 3 fp32 positions in [0, L) (device);
 *   domain_of_atom: n_atoms int32 domain ids (device; trusted, range-checked).
 * Synchronises `stream` once.  On success *out_plan owns device memory until
 * halo_destroy().  Errors: HALO_EINVAL, HALO_EPULSES, HALO_EDOMAIN,
 * HALO_ENOMEM, HALO_ECUDA. */
int halo_setup(const float box[3], const int32_t grid[3], float rc, const float* coords,
               const int32_t* domain_of_atom, int64_t n_atoms, void* stream,
               halo_plan** out_plan);

/* Plan options of halo_setup_ex.
 *   HALO_SETUP_PRUNE_CORNERS: corner pruning of forwarded candidates.  The
 *     page "Redesigning GROMACS Halo Exchange ..." (section 3) selects, per
 *     pulse, the atoms within the cut-off of the neighbour's face (a
 *     one-dimensional slab) and has no counterpart for this option.  With it,
 *     a candidate of a pulse in dim d that passes the face threshold is sent
 *     only if its distance to the receiver's home box, over d and every dim
 *     across whose upper face the slot was received on its forwarding path, is
 *     below rc: in double, max(0, x_d - the sender's lower face)^2 first, then
 *     max(0, x_e - the sender's upper face in e)^2 for those dims e in
 *     ascending order, compared strictly with rc * rc (faces c * L / n in
 *     double).  Every pair within rc that the receiver computes under the
 *     eighth-shell assignment keeps both atoms; only corner and edge atoms
 *     that no such pair needs are dropped, so halos shrink (more in thin
 *     domains and several-pulse dims).  Everything else, including the
 *     exchanges and their modes, is unchanged. */
#define HALO_SETUP_PRUNE_CORNERS 1u

/* halo_setup with options (a bitwise or of HALO_SETUP_* flags; 0 gives
 * halo_setup).  Unknown bits: HALO_EINVAL.  The flags are kept across
 * halo_rebuild and reported by halo_query. */
int halo_setup_ex(const float box[3], const int32_t grid[3], float rc, const float* coords,
                  const int32_t* domain_of_atom, int64_t n_atoms, uint32_t flags, void* stream,
                  halo_plan** out_plan);

/* Rebuild the plan's maps for new positions / domain ids (same box, grid and
 * cut-off; n_atoms may change).  Synchronises `stream`.  Sizes and layout
 * change: query them again and re-size the caller's buffers.  If the rebuild
 * fails, the plan refuses exchanges and the layout, pulse and index-map
 * queries (HALO_EINVAL) until a rebuild succeeds. */
int halo_rebuild(halo_plan* plan, const float* coords, const int32_t* domain_of_atom,
                 int64_t n_atoms, void* stream);

/* Sizes of the plan (host struct). */
int halo_query(const halo_plan* plan, halo_info* out);

/* Dense layout (host arrays of n_domains entries each; any may be NULL). */
int halo_domain_layout(const halo_plan* plan, int64_t* base, int32_t* n_home, int32_t* n_local);

/* One pulse of one sender domain (host struct); if index_map (host) is not
 * NULL it receives send_size int32 entries.  Synchronous copy. */
int halo_get_pulse(const halo_plan* plan, int32_t domain, int32_t pulse, halo_pulse_info* out,
                   int32_t* index_map);

/* All index maps (host): maps receives n_halo_total int32 entries; the map of
 * (sender s, pulse p) is maps[offsets[p*n_domains + s] .. offsets[p*n_domains
 * + s + 1]); offsets (host) has n_pulses*n_domains + 1 entries.  Synchronous. */
int halo_get_index_maps(const halo_plan* plan, int32_t* maps, int64_t* offsets);

/* Global atom id of the owner of every local slot: out has n_local_total
 * int32 (device).  Asynchronous on stream. */
int halo_local_to_global(const halo_plan* plan, int32_t* out, void* stream);

/* Copy the home atoms' coordinates from the global array (n_atoms x 3) into
 * the dense local layout (n_local_total x 3); halo slots are not touched. */
int halo_load_home(const halo_plan* plan, const float* global_xyz, float* local_xyz,
                   void* stream);

/* The inverse of halo_load_home: copy the home slots of the dense local
 * layout (n_local_total x 3, e.g. the forces after halo_exchange_f) back to a
 * global array (n_atoms x 3) in input atom order; halo slots are not read.
 * The pages have no counterpart (their ranks keep their atoms); a caller
 * integrating in input order needs it.  Asynchronous. */
int halo_store_home(const halo_plan* plan, const float* local_xyz, float* global_xyz,
                    void* stream);

/* Coordinate halo exchange (FusedPackCommX, Algorithms 3/4), one kernel
 * launch for all pulses: for every pulse p and sender s,
 *   local_coords[base[r] + atom_offset + i] = local_coords[base[s] + map[i]] + coord_shift,
 * i in [0, send_size).  local_coords: n_local_total x 3 fp32, caller-owned,
 * home slots filled.  Asynchronous. */
int halo_exchange_x(halo_plan* plan, float* local_coords, void* stream);

/* Coordinate exchange that allocates no device memory.  The page has no
 * counterpart: this call exists for callers that may not allocate device
 * memory when they call in (a host framework whose pool allocator owns all
 * device memory, or a latency-critical loop where a cudaMalloc / cudaFree,
 * which can synchronise the whole device, is not acceptable).
 * Same result as halo_exchange_x in HALO_MODE_FUSED, whatever the plan's mode:
 * the same kernel, with its arrival counters and work ticket taken from a
 * fixed array compiled into the library (HALO_NOALLOC_MAX_COUNTERS counters,
 * 64 KiB, held by every GPU that loads the library until exit) instead of the
 * plan's memory.  The plan itself comes from halo_setup.
 *   - The plan needs the FUSED mode's work lists: they exist when its last
 *     setup or rebuild ran in HALO_MODE_FUSED (the default), or after a
 *     halo_set_mode(HALO_MODE_FUSED) since.  Otherwise HALO_EINVAL and
 *     nothing runs (building them would allocate).
 *   - n_domains * n_pulses must be <= HALO_NOALLOC_MAX_COUNTERS, else
 *     HALO_ESCRATCH and nothing runs.
 *   - halo_setup looks the array's device address up (cudaGetSymbolAddress,
 *     once per device, with that device current); under lazy module loading
 *     that is when the array is placed in device memory.  This call only
 *     reads the stored address, so even the first call on a device loads and
 *     allocates nothing.  HALO_ECUDA if no address is stored for the plan's
 *     device.
 *   - Each call clears the part of the array it uses (an asynchronous memset
 *     on `stream`) before its launch.  All calls share the array: calls whose
 *     kernels overlap on the GPU race and give wrong results.
 * Asynchronous; a timed-out wait is reported by halo_status() as usual. */
#define HALO_NOALLOC_MAX_COUNTERS 16384
int halo_exchange_x_noalloc(halo_plan* plan, float* local_coords, void* stream);

/* Force halo reduction (FusedCommUnpackF, Algorithm 6), one kernel launch for
 * all pulses: for p = P-1 .. 0 and every sender s,
 *   local_forces[base[s] + map[i]] += local_forces[base[r] + atom_offset + i].
 * Halo slots keep their (possibly forwarded-into) values.  Bit-identical to
 * the sequential order.  Asynchronous. */
int halo_exchange_f(halo_plan* plan, float* local_forces, void* stream);

/* ---- Sharded data plane ------------------------------------------------------
 * The page "Redesigning GROMACS Halo Exchange ..." spreads the domains over
 * several GPUs: a pulse whose receiver sits on another GPU stores the packed
 * coordinates into that GPU's halo slice and signals it with a system-scope
 * release (section 3, NVLink path; section 4, memory ordering), and the force
 * pass reads the remote halo forces back (Algorithm 6).  These calls split a
 * plan's domains into n_shards z-slabs, each with its own buffer, and run the
 * FUSED exchanges across them with system-scope signals.  In one process on
 * one GPU every shard's work runs in one launch per direction.
 *
 * Shard k holds the domains [first_domain, first_domain + n_domains) (domain
 * id = ix + nx*(iy + ny*iz), so a z-slab is a contiguous id range), laid out
 * as in the dense local array: domain by domain, [home | halo of pulse 0 | ...].
 * Its buffer holds n_local x 3 fp32 (caller-owned); the dense slot g of the
 * plan is slot g - first_slot of its shard's buffer.
 *
 * halo_shard: n_shards in [1, min(HALO_MAX_SHARDS, n_z)], shard k taking the
 *   z layers [k*nz/n_shards, (k+1)*nz/n_shards).  Builds the FUSED work lists
 *   with each item's source and destination shard (synchronises `stream`).
 *   The partition persists across halo_rebuild (which then rebuilds those
 *   lists whatever the mode).  HALO_EINVAL for a bad count.
 * halo_shard_layout: shard k's domains and slots (host outputs, nullable).
 * halo_load_home_sharded / halo_store_home_sharded: halo_load_home /
 *   halo_store_home with the local array split into the shards' buffers.
 * halo_exchange_x_sharded / halo_exchange_f_sharded: halo_exchange_x /
 *   halo_exchange_f in HALO_MODE_FUSED on the shards' buffers (an array of
 *   n_shards device pointers, host memory, read during the call): the same
 *   result bit for bit, whatever the plan's mode.  HALO_EINVAL for a null or
 *   misaligned buffer pointer or a plan without FUSED work lists.
 *   Asynchronous; timeouts are reported by halo_status() as usual. */
int halo_shard(halo_plan* plan, int32_t n_shards, void* stream);
int halo_shard_layout(const halo_plan* plan, int32_t shard, int32_t* first_domain /*host*/,
                      int32_t* n_domains /*host*/, int64_t* first_slot /*host*/,
                      int64_t* n_local /*host*/);
int halo_load_home_sharded(const halo_plan* plan, const float* global_xyz,
                           float* const* shard_local /*host array of device pointers*/, void* stream);
int halo_store_home_sharded(const halo_plan* plan, const float* const* shard_local /*host array*/,
                            float* global_xyz, void* stream);
int halo_exchange_x_sharded(halo_plan* plan, float* const* shard_coords /*host array*/, void* stream);
int halo_exchange_f_sharded(halo_plan* plan, float* const* shard_forces /*host array*/, void* stream);

/* Select how halo_exchange_x / halo_exchange_f run (HALO_MODE_*).
 *   FUSED: the pages' design (Algorithms 3-6): one launch per direction; the
 *     entries below depOffset stream at once, forwarded entries wait on
 *     per-(domain, pulse) release/acquire counters.
 *   STEPWISE: one launch per pulse and direction (the pages' first design,
 *     one kernel per pulse ordered by the stream); P launches per call.
 *   STAGED: the GPU-aware-MPI schedule the page "GPU-Initiated Halo Exchange
 *     Cuts CPU Bottlenecks in GROMACS" starts from (section "The CPU
 *     bottleneck in halo exchange"): per pulse a pack kernel into a send
 *     buffer, a host wait, a transfer kernel standing in for the MPI
 *     messages of all domains, a host wait (forces: transfer, wait, unpack
 *     kernel, wait; last pulse first).  2P launches and 2P stream
 *     synchronisations per call, so the calls block the host and cannot be
 *     captured in a CUDA graph.  Needs a buffer of 12 bytes per halo slot
 *     (allocated here and by halo_rebuild).
 *   FLAT: every halo slot's forwarding chain composed at build time (owner,
 *     periodic shift; per owner the tree of its copies in reverse creation
 *     order); one launch per direction with no waits.  Needs extra tables
 *     (built here, synchronising `stream`; rebuilt by halo_rebuild) and
 *     n_local_total < 2^26, at most 63 copies per atom (HALO_ECAPACITY
 *     otherwise).
 * The mode is kept across halo_rebuild.  A setup or rebuild builds the
 * tables of the plan's current mode only; selecting FUSED or FLAT later
 * builds theirs (synchronising `stream`).  HALO_EINVAL on a plan whose last
 * rebuild failed when the selected mode's tables would have to be built. */
int halo_set_mode(halo_plan* plan, int32_t mode, void* stream);
int halo_get_mode(const halo_plan* plan, int32_t* mode);

/* Synchronise `stream`, return the plan's sticky device error (HALO_OK if
 * none) and clear it, resetting the plan's flags. */
int halo_status(halo_plan* plan, void* stream);

/* Test hook: the next halo_rebuild starts with a build buffer of `slots`
 * slots (> 0; never fewer than the home atoms + 1) instead of its geometric
 * estimate.  If that is too small, the build overflows, detects it and
 * retries with a larger buffer (see halo_info.build_attempts).  The device
 * kernels never write past the buffer they were given. */
int halo_debug_set_build_capacity(halo_plan* plan, int64_t slots);

/* Time limit of every device-side wait.  seconds > 0.  The default of a new
 * plan is 1 s, or HALO_WAIT_TIMEOUT_MS milliseconds when that environment
 * variable holds a positive number at halo_setup. */
int halo_set_wait_timeout(halo_plan* plan, double seconds);

/* The words a setup or rebuild reads back (sizes, counts, errors) are written
 * by its last kernels straight into the plan's pinned host staging, mapped
 * into the device's address space.  Where that staging cannot be mapped, or
 * when the environment variable HALO_STAGE_COPIES is set (not "0") at
 * halo_setup, they are copied back instead; the results are the same. */

/* Test hook: in the next halo_exchange_x, the producer of (domain, pulse)
 * skips its completion signal, so its consumers' waits run out and the kernel
 * reports HALO_ETIMEOUT through halo_status().  (-1, -1) disarms. */
int halo_debug_drop_signal(halo_plan* plan, int32_t domain, int32_t pulse);

/* Tracing (optional).  trace: device buffer of 4 * capacity_items uint64
 * words, caller-owned; capacity_items >= x_items + f_items of
 * halo_work_items().  While armed, every work item of both exchange kernels
 * records {time it was taken, time its waits ended, time it released its
 * signal (global timer, ns), SM id}: coordinate items at [0, x_items), force
 * items after them.  NULL disarms; a rebuild disarms.  HALO_EINVAL while
 * the plan has no FUSED work lists.  For diagnosis only. */
int halo_set_trace(halo_plan* plan, uint64_t* trace, int64_t capacity_items);

/* Work decomposition of the FUSED exchanges (host): items per kernel, entries
 * per item; HALO_EINVAL while the plan has no FUSED work lists. */
int halo_work_items(const halo_plan* plan, int32_t* x_items, int32_t* f_items, int32_t* chunk);

/* Kernel launches made so far by halo_exchange_x and halo_exchange_f (host). */
int halo_launch_counts(const halo_plan* plan, int64_t* x_launches, int64_t* f_launches);

void halo_destroy(halo_plan* plan);

const char* halo_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* HALO_H */
