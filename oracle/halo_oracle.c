/*
 * halo_oracle.c -- plain, sequential CPU oracle for the eighth-shell
 * domain-decomposition halo exchange.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the reference the CUDA library's
 * results are compared against.  Only the tests, __graft_entry__.smoke() and the
 * cpu_baseline / --impl reference legs of bench.py may load it.  It shares no
 * code, header, table or helper with the CUDA library and must never be
 * reached from the library's product path.
 *
 * What it follows (page: "Redesigning GROMACS Halo Exchange: Improving Strong
 * Scaling with GPU-initiated NVSHMEM", paper review):
 *   - section 3 "GROMACS domain-decomposition halo exchange": neutral-territory
 *     decomposition, each domain owns its home atoms; boundary atoms within the
 *     cut-off are forwarded through intermediate domains (eighth shell), with
 *     np(z) pulses in z, then np(y) in y, then np(x) in x;
 *   - Algorithm 1 (PulseData: sendRank, recvRank, sendSize, recvSize,
 *     atomOffset, coordShift, indexMap);
 *   - Algorithm 4 (packWithDeps: entries with indexMap[i] < depOffset are
 *     independent, the rest were received in earlier pulses) and the
 *     "global pulse order Z -> Y -> X" paragraph after it;
 *   - Algorithm 6 (FusedCommUnpackF: pulses from the last down to 0, each
 *     received force entry added to the atom its index-map entry names).
 *
 * Readings of what the page leaves open (each one is also listed in the
 * design notes):
 *   R1  domain id D = ix + nx*(iy + ny*iz); w_d = L_d/n_d (double);
 *       p_d = ceil(rc/w_d) pulses in a decomposed dim (n_d > 1), 0 otherwise;
 *       p_d >= n_d is rejected (the halo would wrap onto its own domain).
 *   R2  coordinates flow from sender s to receiver r = s - e_d (periodic):
 *       every domain's halo lies above its upper faces.
 *   R3  predicate: x'_d < thr_d(s), one fp32 compare, strict, with
 *       thr_d(s) = fl32(s_d * L_d / n_d + rc) evaluated in double.
 *   R4  candidates of pulse k of dim d: k == 0 -> local slots [0, atomOffset
 *       of this pulse) (home plus all halo of earlier dims); k >= 1 -> only the
 *       slots received in pulse k-1 of the same dim.
 *   R5  indexMap entries ascending by local index; depOffset = n_home[s];
 *       split = number of entries < depOffset.
 *   R6  coordShift: +L_d on component d iff s_d == 0, else 0; the shifted
 *       coordinate is one fp32 add per component.
 *   R7  force reduction: pulses P-1 ... 0; plain add (entries are unique
 *       within a pulse); halo force slots keep whatever they hold.
 *   R8  optional corner pruning (off unless asked for; the page describes
 *       one-dimensional face slabs only): a candidate that passes R3 is kept
 *       only if its distance to the receiver's home box, over the dims in
 *       which it is beyond that box, is below rc.  The dims are d itself (the
 *       distance past the receiver's upper face, which is the sender's lower
 *       face) and every dim across whose upper face the slot was received on
 *       its way to the sender (its forwarding path).  In double: each term
 *       max(0, x - face) squared, d's term first and then the other dims in
 *       ascending order, compared strictly with rc * rc; faces c * L / n in
 *       double as in R3.  No pair within rc that the receiver computes (both
 *       atoms inside its home slab in every dim where either is beyond it, the
 *       eighth-shell assignment) loses an atom: the partner lies inside the
 *       box in those dims, so their distance is at least this one.
 *
 * Build: gcc -std=c11 -O2 -fno-fast-math -ffp-contract=off -shared -fPIC
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_EPULSES (-2)
#define ORC_EDOMAIN (-3)
#define ORC_ENOMEM (-4)
#define ORC_MAX_PULSES 64

typedef struct {
    int32_t *v;
    int64_t n, cap;
} ivec;

typedef struct {
    float *v; /* xyz triples */
    int64_t n, cap; /* counted in atoms */
} fvec3;

typedef struct {
    /* problem */
    int grid[3];
    float box[3];
    float rc;
    int64_t n_atoms;
    int n_dom;
    /* pulses in global order */
    int pulses_per_dim[3];
    int n_pulses;
    int pulse_dim[ORC_MAX_PULSES];
    int pulse_k[ORC_MAX_PULSES]; /* index of the pulse within its dim */
    /* per domain */
    int32_t *n_home;
    int32_t *n_local;
    int64_t *base; /* first slot of the domain in the dense local layout */
    fvec3 *xyz;    /* local coordinates built at setup (home + halo) */
    ivec *gid;     /* global atom id of the owner of each local slot */
    /* per (sender s, pulse p), flat index s * n_pulses + p */
    int32_t *recv_dom;
    int32_t *send_size;
    int32_t *split;
    int32_t *atom_offset; /* first slot of this pulse's halo in the receiver */
    float *shift;         /* 3 per (s, p) */
    ivec *map;
    int prune;   /* reading R8 */
    ivec *disp;  /* per domain and local slot: bit e set iff the slot was received
                    across an upper face in dim e (on its whole forwarding path) */
    int threads; /* exchanges: OpenMP threads over the domains of one pulse (<= 1: none) */
} oracle_t;

static int ivec_push(ivec *a, int32_t x)
{
    if (a->n == a->cap) {
        int64_t nc = a->cap ? 2 * a->cap : 64;
        int32_t *nv = (int32_t *)realloc(a->v, (size_t)nc * sizeof(int32_t));
        if (!nv) return ORC_ENOMEM;
        a->v = nv;
        a->cap = nc;
    }
    a->v[a->n++] = x;
    return ORC_OK;
}

static int fvec3_push(fvec3 *a, float x, float y, float z)
{
    if (a->n == a->cap) {
        int64_t nc = a->cap ? 2 * a->cap : 64;
        float *nv = (float *)realloc(a->v, (size_t)nc * 3 * sizeof(float));
        if (!nv) return ORC_ENOMEM;
        a->v = nv;
        a->cap = nc;
    }
    a->v[3 * a->n + 0] = x;
    a->v[3 * a->n + 1] = y;
    a->v[3 * a->n + 2] = z;
    a->n++;
    return ORC_OK;
}

void oracle_free(oracle_t *o)
{
    if (!o) return;
    if (o->xyz)
        for (int d = 0; d < o->n_dom; d++) free(o->xyz[d].v);
    if (o->gid)
        for (int d = 0; d < o->n_dom; d++) free(o->gid[d].v);
    if (o->disp)
        for (int d = 0; d < o->n_dom; d++) free(o->disp[d].v);
    if (o->map)
        for (int i = 0; i < o->n_dom * o->n_pulses; i++) free(o->map[i].v);
    free(o->xyz);
    free(o->gid);
    free(o->disp);
    free(o->map);
    free(o->n_home);
    free(o->n_local);
    free(o->base);
    free(o->recv_dom);
    free(o->send_size);
    free(o->split);
    free(o->atom_offset);
    free(o->shift);
    free(o);
}

/* Cell coordinates of domain id D (reading R1). */
static void domain_cell(const oracle_t *o, int D, int c[3])
{
    c[0] = D % o->grid[0];
    c[1] = (D / o->grid[0]) % o->grid[1];
    c[2] = D / (o->grid[0] * o->grid[1]);
}

static int domain_id(const oracle_t *o, const int c[3])
{
    return c[0] + o->grid[0] * (c[1] + o->grid[1] * c[2]);
}

/* Reading R8: is local slot i of sender s (cell c), a candidate of a pulse in
 * dim d, within rc of the receiver's home box over the dims where it lies
 * beyond it? */
static int within_corner(const oracle_t *o, int s, const int c[3], int d, int32_t i)
{
    const float *x = &o->xyz[s].v[3 * (int64_t)i];
    const int32_t m = o->disp[s].v[i];
    const double lo_d = (double)c[d] * (double)o->box[d] / (double)o->grid[d];
    double t = (double)x[d] - lo_d;
    if (t < 0.0) t = 0.0;
    double r2 = t * t;
    for (int e = 0; e < 3; e++) {
        if (e == d || !((m >> e) & 1)) continue;
        const double hi_e = (double)(c[e] + 1) * (double)o->box[e] / (double)o->grid[e];
        double u = (double)x[e] - hi_e;
        if (u < 0.0) u = 0.0;
        r2 = r2 + u * u;
    }
    return r2 < (double)o->rc * (double)o->rc;
}

int oracle_setup_ex(const float box[3], const int grid[3], float rc,
                    const float *xyz, const int32_t *dom, int64_t n_atoms,
                    int flags, oracle_t **out);

int oracle_setup(const float box[3], const int grid[3], float rc,
                 const float *xyz, const int32_t *dom, int64_t n_atoms,
                 oracle_t **out)
{
    return oracle_setup_ex(box, grid, rc, xyz, dom, n_atoms, 0, out);
}

/* flags: 1 = corner pruning (reading R8). */
int oracle_setup_ex(const float box[3], const int grid[3], float rc,
                    const float *xyz, const int32_t *dom, int64_t n_atoms,
                    int flags, oracle_t **out)
{
    *out = NULL;
    if (!box || !grid || !xyz || !dom || n_atoms <= 0) return ORC_EINVAL;
    if (!(rc > 0.0f)) return ORC_EINVAL;
    for (int d = 0; d < 3; d++)
        if (grid[d] < 1 || !(box[d] > 0.0f)) return ORC_EINVAL;

    oracle_t *o = (oracle_t *)calloc(1, sizeof(oracle_t));
    if (!o) return ORC_ENOMEM;
    for (int d = 0; d < 3; d++) {
        o->grid[d] = grid[d];
        o->box[d] = box[d];
    }
    o->rc = rc;
    o->prune = (flags & 1) != 0;
    o->n_atoms = n_atoms;
    o->n_dom = grid[0] * grid[1] * grid[2];

    /* Step 1: pulses per dim and the global order z..., y..., x...
     * (section 3: np(z) pulses in z, then np(y) in y, then np(x) in x). */
    for (int d = 0; d < 3; d++) {
        int p = 0;
        if (grid[d] > 1) {
            double w = (double)box[d] / (double)grid[d];
            p = (int)ceil((double)rc / w);
        }
        if (p >= grid[d] && grid[d] > 1) {
            oracle_free(o);
            return ORC_EPULSES;
        }
        o->pulses_per_dim[d] = p;
    }
    o->n_pulses = 0;
    for (int d = 2; d >= 0; d--) {
        for (int k = 0; k < o->pulses_per_dim[d]; k++) {
            if (o->n_pulses >= ORC_MAX_PULSES) {
                oracle_free(o);
                return ORC_EINVAL;
            }
            o->pulse_dim[o->n_pulses] = d;
            o->pulse_k[o->n_pulses] = k;
            o->n_pulses++;
        }
    }
    const int P = o->n_pulses;
    const int ND = o->n_dom;

    for (int64_t a = 0; a < n_atoms; a++)
        if (dom[a] < 0 || dom[a] >= ND) {
            oracle_free(o);
            return ORC_EDOMAIN;
        }

    o->n_home = (int32_t *)calloc((size_t)ND, sizeof(int32_t));
    o->n_local = (int32_t *)calloc((size_t)ND, sizeof(int32_t));
    o->base = (int64_t *)calloc((size_t)ND, sizeof(int64_t));
    o->xyz = (fvec3 *)calloc((size_t)ND, sizeof(fvec3));
    o->gid = (ivec *)calloc((size_t)ND, sizeof(ivec));
    o->disp = (ivec *)calloc((size_t)ND, sizeof(ivec));
    size_t nsp = (size_t)ND * (size_t)(P > 0 ? P : 1);
    o->recv_dom = (int32_t *)calloc(nsp, sizeof(int32_t));
    o->send_size = (int32_t *)calloc(nsp, sizeof(int32_t));
    o->split = (int32_t *)calloc(nsp, sizeof(int32_t));
    o->atom_offset = (int32_t *)calloc(nsp, sizeof(int32_t));
    o->shift = (float *)calloc(3 * nsp, sizeof(float));
    o->map = (ivec *)calloc(nsp, sizeof(ivec));
    if (!o->n_home || !o->n_local || !o->base || !o->xyz || !o->gid || !o->disp ||
        !o->recv_dom || !o->send_size || !o->split || !o->atom_offset ||
        !o->shift || !o->map) {
        oracle_free(o);
        return ORC_ENOMEM;
    }

    /* Step 2: home atoms of each domain, in input order (ownership by
     * domain, section 3). */
    for (int64_t a = 0; a < n_atoms; a++) {
        int D = dom[a];
        if (fvec3_push(&o->xyz[D], xyz[3 * a], xyz[3 * a + 1], xyz[3 * a + 2]) ||
            ivec_push(&o->gid[D], (int32_t)a) || ivec_push(&o->disp[D], 0)) {
            oracle_free(o);
            return ORC_ENOMEM;
        }
        o->n_home[D]++;
    }

    /* Step 3: the pulses, in global order.  Each pulse is computed from the
     * state at its start: first every sender's index map, then every
     * receiver's new halo slots. */
    int32_t *cand_lo = (int32_t *)malloc((size_t)ND * sizeof(int32_t));
    int32_t *cand_hi = (int32_t *)malloc((size_t)ND * sizeof(int32_t));
    int32_t *prev_start = (int32_t *)malloc((size_t)ND * sizeof(int32_t));
    if (!cand_lo || !cand_hi || !prev_start) {
        free(cand_lo);
        free(cand_hi);
        free(prev_start);
        oracle_free(o);
        return ORC_ENOMEM;
    }
    for (int p = 0; p < P; p++) {
        const int d = o->pulse_dim[p];
        const int k = o->pulse_k[p];
        for (int s = 0; s < ND; s++) {
            /* reading R4: candidate slots of sender s */
            cand_hi[s] = (int32_t)o->xyz[s].n;
            cand_lo[s] = (k == 0) ? 0 : prev_start[s];
        }
        for (int s = 0; s < ND; s++) {
            int c[3];
            domain_cell(o, s, c);
            int rc3[3] = {c[0], c[1], c[2]};
            rc3[d] = (c[d] - 1 + o->grid[d]) % o->grid[d]; /* reading R2 */
            const int r = domain_id(o, rc3);
            const int sp = s * P + p;
            /* reading R3: threshold = lower face of s plus the cut-off */
            const float thr = (float)((double)c[d] * (double)box[d] /
                                          (double)grid[d] +
                                      (double)rc);
            ivec *m = &o->map[sp];
            for (int32_t i = cand_lo[s]; i < cand_hi[s]; i++) {
                if (o->xyz[s].v[3 * (int64_t)i + d] < thr &&
                    (!o->prune || within_corner(o, s, c, d, i))) {
                    if (ivec_push(m, i)) {
                        free(cand_lo);
                        free(cand_hi);
                        free(prev_start);
                        oracle_free(o);
                        return ORC_ENOMEM;
                    }
                }
            }
            o->recv_dom[sp] = r;
            o->send_size[sp] = (int32_t)m->n;
            int32_t nsplit = 0; /* reading R5, Algorithm 4 depOffset */
            for (int64_t j = 0; j < m->n; j++)
                if (m->v[j] < o->n_home[s]) nsplit++;
            o->split[sp] = nsplit;
            for (int e = 0; e < 3; e++) o->shift[3 * sp + e] = 0.0f;
            if (c[d] == 0) o->shift[3 * sp + d] = box[d]; /* reading R6 */
        }
        /* receivers append the new halo: coordinate + coordShift */
        for (int s = 0; s < ND; s++) {
            const int sp = s * P + p;
            const int r = o->recv_dom[sp];
            const ivec *m = &o->map[sp];
            const float *sh = &o->shift[3 * sp];
            o->atom_offset[sp] = (int32_t)o->xyz[r].n;
            prev_start[r] = (int32_t)o->xyz[r].n;
            for (int64_t j = 0; j < m->n; j++) {
                const float *src = &o->xyz[s].v[3 * (int64_t)m->v[j]];
                if (fvec3_push(&o->xyz[r], src[0] + sh[0], src[1] + sh[1],
                               src[2] + sh[2]) ||
                    ivec_push(&o->gid[r], o->gid[s].v[m->v[j]]) ||
                    ivec_push(&o->disp[r], o->disp[s].v[m->v[j]] | (1 << d))) {
                    free(cand_lo);
                    free(cand_hi);
                    free(prev_start);
                    oracle_free(o);
                    return ORC_ENOMEM;
                }
            }
        }
    }
    free(cand_lo);
    free(cand_hi);
    free(prev_start);

    /* dense layout: base[D] = sum of local sizes of lower domain ids */
    int64_t acc = 0;
    for (int D = 0; D < ND; D++) {
        o->n_local[D] = (int32_t)o->xyz[D].n;
        o->base[D] = acc;
        acc += o->n_local[D];
    }
    *out = o;
    return ORC_OK;
}

/* ---- accessors ---------------------------------------------------------- */

int oracle_num_domains(const oracle_t *o) { return o->n_dom; }
int oracle_num_pulses(const oracle_t *o) { return o->n_pulses; }

void oracle_pulses(const oracle_t *o, int32_t *per_dim3, int32_t *dims)
{
    for (int d = 0; d < 3; d++) per_dim3[d] = o->pulses_per_dim[d];
    for (int p = 0; p < o->n_pulses; p++) dims[p] = o->pulse_dim[p];
}

int64_t oracle_n_local_total(const oracle_t *o)
{
    int64_t t = 0;
    for (int D = 0; D < o->n_dom; D++) t += o->n_local[D];
    return t;
}

void oracle_layout(const oracle_t *o, int64_t *base, int32_t *n_home,
                   int32_t *n_local)
{
    for (int D = 0; D < o->n_dom; D++) {
        base[D] = o->base[D];
        n_home[D] = o->n_home[D];
        n_local[D] = o->n_local[D];
    }
}

/* info: send_domain, recv_domain, send_size, split, dep_offset, atom_offset */
int oracle_pulse_info(const oracle_t *o, int s, int p, int32_t info[6],
                      float shift[3])
{
    if (s < 0 || s >= o->n_dom || p < 0 || p >= o->n_pulses) return ORC_EINVAL;
    const int sp = s * o->n_pulses + p;
    info[0] = s;
    info[1] = o->recv_dom[sp];
    info[2] = o->send_size[sp];
    info[3] = o->split[sp];
    info[4] = o->n_home[s];
    info[5] = o->atom_offset[sp];
    for (int e = 0; e < 3; e++) shift[e] = o->shift[3 * sp + e];
    return ORC_OK;
}

int oracle_index_map(const oracle_t *o, int s, int p, int32_t *out)
{
    if (s < 0 || s >= o->n_dom || p < 0 || p >= o->n_pulses) return ORC_EINVAL;
    const ivec *m = &o->map[s * o->n_pulses + p];
    if (m->n) memcpy(out, m->v, (size_t)m->n * sizeof(int32_t));
    return ORC_OK;
}

/* Local coordinates as built at setup, dense layout (n_local_total x 3). */
void oracle_local_coords(const oracle_t *o, float *out)
{
    for (int D = 0; D < o->n_dom; D++)
        memcpy(out + 3 * o->base[D], o->xyz[D].v,
               (size_t)o->n_local[D] * 3 * sizeof(float));
}

/* Global atom id of the owner of every local slot, dense layout. */
void oracle_local_to_global(const oracle_t *o, int32_t *out)
{
    for (int D = 0; D < o->n_dom; D++)
        memcpy(out + o->base[D], o->gid[D].v,
               (size_t)o->n_local[D] * sizeof(int32_t));
}

/* Home coordinates from global arrays into the dense local layout. */
void oracle_load_home(const oracle_t *o, const float *global_xyz, float *local)
{
    for (int D = 0; D < o->n_dom; D++)
        for (int32_t j = 0; j < o->n_home[D]; j++) {
            const int64_t a = o->gid[D].v[j];
            for (int e = 0; e < 3; e++)
                local[3 * (o->base[D] + j) + e] = global_xyz[3 * a + e];
        }
}

/* Host threads for the two exchanges (default: none).  The senders of one
 * pulse are independent.  Coordinates: a sender writes only its receiver's
 * slots of this pulse (each receiver has one sender per pulse) and reads only
 * slots filled before this pulse.  Forces: a sender adds into its own mapped
 * slots, which are home or earlier-pulse slots that no other sender of the
 * pulse touches, from its receiver's slots of this pulse, which no sender of
 * the pulse writes.  So running the senders of a pulse on several threads
 * changes neither a value nor the order of the adds into any slot; pulses stay
 * in sequence. */
void oracle_set_threads(oracle_t *o, int threads)
{
    o->threads = threads;
}

int oracle_openmp(void)
{
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}

/* Coordinate halo exchange on the dense local layout: for every pulse in
 * order and every sender, gather the index-mapped slots, add coordShift and
 * write them to the receiver's halo slots (Algorithms 3 and 4). */
void oracle_exchange_x(const oracle_t *o, float *local)
{
    const int P = o->n_pulses;
    const int nt = o->threads > 1 ? o->threads : 1;
    for (int p = 0; p < P; p++)
#pragma omp parallel for schedule(static) if (nt > 1) num_threads(nt)
        for (int s = 0; s < o->n_dom; s++) {
            const int sp = s * P + p;
            const ivec *m = &o->map[sp];
            const int r = o->recv_dom[sp];
            const float *sh = &o->shift[3 * sp];
            float *dst = local + 3 * (o->base[r] + o->atom_offset[sp]);
            const float *src = local + 3 * o->base[s];
            for (int64_t i = 0; i < m->n; i++)
                for (int e = 0; e < 3; e++)
                    dst[3 * i + e] = src[3 * (int64_t)m->v[i] + e] + sh[e];
        }
}

/* Force halo reduction on the dense local layout: pulses from the last to
 * the first; the receiver's halo force of entry i is added to the sender's
 * slot indexMap[i] (Algorithm 6). */
void oracle_exchange_f(const oracle_t *o, float *local)
{
    const int P = o->n_pulses;
    const int nt = o->threads > 1 ? o->threads : 1;
    for (int p = P - 1; p >= 0; p--)
#pragma omp parallel for schedule(static) if (nt > 1) num_threads(nt)
        for (int s = 0; s < o->n_dom; s++) {
            const int sp = s * P + p;
            const ivec *m = &o->map[sp];
            const int r = o->recv_dom[sp];
            const float *halo = local + 3 * (o->base[r] + o->atom_offset[sp]);
            float *own = local + 3 * o->base[s];
            for (int64_t i = 0; i < m->n; i++)
                for (int e = 0; e < 3; e++)
                    own[3 * (int64_t)m->v[i] + e] =
                        own[3 * (int64_t)m->v[i] + e] + halo[3 * i + e];
        }
}
