/*
 * bs.h -- C ABI of the GB300 Benchmark Streaming library (libbs.so).
 *
 * The seven Benchmark Streaming (BS) operations of a conjugate-gradient
 * iteration of a high-order spectral-element solver on hexahedral meshes,
 * in IEEE binary64 on one NVIDIA GB300 (sm_103a):
 *
 *   BS1 copy, BS2 AXPY, BS3 norm, BS4 inner product, BS5 fused CG update,
 *   BS6 gather (q_G = Z^T q_L), BS7 scatter (q_L = Z q_G),
 *
 * as defined in "Portable high-order finite element kernels I: Streaming
 * Operations" (the Benchmark Streaming test list; the CG vector operations;
 * eq. (3) v_L = Z v_G; the gather/scatter kernel descriptions), plus the
 * box-mesh index tables they run on and the sequence of one CG iteration.
 *
 * Conventions for every call below:
 *  - Vectors are contiguous binary64 arrays in DEVICE memory, owned by the
 *    caller (for instance torch tensors).  The library never allocates in
 *    an operation call; its only device allocation is the small reduction
 *    workspace of a context, made by bs_ctx_create.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL is the legacy default stream).  Results are valid once the stream
 *    has reached the call's position.
 *  - Scalars a reduction produces are written to device memory (`*_dev`).
 *  - The device current on the calling thread must be the context's device.
 *  - Lengths are int64_t; index tables are int32_t (at most 2^31 - 1
 *    entries).  n == 0 is a no-op, except that a reduction of length 0
 *    writes +0.0.
 *  - Pointers need only binary64 alignment (8 bytes).  The kernels peel a
 *    misaligned head so that the bulk runs with 32-byte vectors; when the
 *    operands are misaligned relative to each other a narrower vector width
 *    is used.  BS_EALIGN is therefore never returned.
 *  - Reductions are deterministic: for a given context (device), length
 *    and operand alignment the result is bitwise the same on every run.
 *  - One context serves one stream at a time: its reduction workspace is
 *    shared by all reductions launched through it.  Use one context per
 *    concurrently used stream.
 *  - Return value: BS_OK (0) or a negative status; bs_strerror() names it
 *    and bs_last_error() gives the context's last message.  On an error
 *    nothing is launched.
 */
#ifndef BS_H
#define BS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define BS_OK 0
#define BS_EINVAL (-1)  /* bad argument: NULL pointer, negative length, overlap, ... */
#define BS_ECUDA (-2)   /* a CUDA runtime call or launch failed                     */
#define BS_ENOMEM (-3)  /* host or context workspace allocation failed             */
#define BS_EBOUNDS (-4) /* an index table entry is out of range (host or device)    */
#define BS_EALIGN (-5)  /* reserved; never returned (misalignment is peeled)       */
#define BS_ETIMEOUT (-6) /* a bounded device-side wait gave up (see bs_ctx_device_status) */

/* With a plan, bs_scatter reading a q_G of at most BS_ONEPASS_SCATTER_BYTES
 * and bs_gather reading a q_L of at most BS_ONEPASS_GATHER_BYTES run the
 * one-pass kernels (one launch instead of two): faster where the randomly
 * read vector stays in L2. */
#define BS_ONEPASS_SCATTER_BYTES (32ll << 20)
#define BS_ONEPASS_GATHER_BYTES (8ll << 20)

/* Host-side fault injection, to test a caller's error handling without
 * faulting a GPU: the environment variable BS_FAULT holds a comma-separated
 * list of "alloc" (bs_ctx_create reports BS_ENOMEM), "launch" (every call
 * that would launch work reports BS_ECUDA and launches nothing) and
 * "badtable" (the mesh builders corrupt one scatterIds and one localIds
 * entry after building: bs_mesh_validate reports BS_EBOUNDS, and the
 * one-pass kernels skip the entries and raise the device flag).  Read at
 * every call; unset means no faults. */

/* ---- mesh flags (bs_mesh_build_box) ------------------------------------- */
#define BS_MESH_SHUFFLE_ELEMS 1u   /* seeded random order of elements in storage */
#define BS_MESH_PERMUTE_GLOBAL 2u  /* seeded random global node numbering        */
#define BS_MESH_MASK_BOUNDARY 4u   /* boundary local nodes get id -1 (masked)    */
#define BS_MESH_ROTATE_ELEMS 8u    /* seeded random orientation of every element */

/* Largest number of CSR entries in one gather row segment the gather kernel
 * can stage in shared memory. */
#define BS_GATHER_SEG_MAX 4096
/* Default target number of CSR entries per gather row segment. */
#define BS_GATHER_SEG_DEFAULT 2048

typedef struct bs_ctx bs_ctx;
typedef struct bs_mesh bs_mesh;

/* Sizes of a built mesh. */
typedef struct {
    int32_t E, N;        /* elements per axis, polynomial degree              */
    uint32_t flags;      /* BS_MESH_* flags it was built with                 */
    int32_t max_row;     /* largest number of local copies of a global node   */
    int64_t K;           /* elements, E^3                                     */
    int64_t NL;          /* local nodes, K (N+1)^3                            */
    int64_t NG;          /* global nodes, (E N + 1)^3                         */
    int64_t nnz;         /* unmasked local nodes = CSR entries of Z^T         */
    int64_t nblocks;     /* gather row segments                               */
    int32_t seg_max;     /* largest number of CSR entries in one segment      */
    int32_t seg_target;  /* target entries per segment it was built with      */
} bs_mesh_info_t;

/* Device copy of a mesh's index tables, as bs_gather / bs_scatter read them.
 * The caller uploads the four host tables of bs_mesh_tables() to device
 * memory it owns and fills in this struct (the struct itself is host
 * memory and is read only during the call).
 *   scatterIds[NL]       local -> global id, -1 = masked       (BS7)
 *   rowStarts[NG+1]      CSR row starts of Z^T, rows = global ids
 *   localIds[nnz]        CSR column (local) ids, ascending within a row
 *   blockStarts[nblocks+1] first row of each gather segment      (BS6) */
/* Two-pass gather/scatter plan in device memory (see bs_mesh_plan below).
 * All table pointers are device memory uploaded by the caller from
 * bs_mesh_plan_tables(); `work` is caller-owned device scratch of at least
 * nnz binary64 values, overwritten by every bs_gather / bs_scatter call
 * that uses the plan (so two such calls must not overlap on the GPU).
 * Sizes are per thread block; a tile or bucket is `cluster` blocks. */
typedef struct {
    int32_t cluster;
    int32_t s_ntiles, s_nbuckets, s_tile_rows, s_bucket_len;
    int32_t g_ntiles, g_nbuckets, g_tile_len, g_bucket_entries_max;
    int32_t g_bucket_rows_max, g_mmax;
    const int32_t *s_tileRows;   /* [s_ntiles+1]                    */
    const int32_t *s_runStart;   /* [(s_ntiles+1) * s_nbuckets]     */
    const uint16_t *s_src;       /* [nnz] bit 15: first slot of a run */
    const uint16_t *s_dst;       /* [nnz]                           */
    const int32_t *g_subRows;    /* [cluster * g_nbuckets + 1]      */
    const int32_t *g_tileSlot;   /* [g_ntiles+1]                    */
    const int32_t *g_runStart;   /* [(g_ntiles+1) * g_nbuckets]     */
    const uint16_t *g_src;       /* [nnz] bit 15: first slot of a run */
    const uint16_t *g_pos;       /* [nnz]                           */
    const uint16_t *g_groupStart; /* [cluster*g_nbuckets*(g_mmax+1)] */
    const uint16_t *g_rowPos;    /* [NG]                            */
    double *work;                /* [work_len >= nnz] scratch (2 nnz for bs_apply_diag) */
    int64_t work_len;
} bs_plan_dev;

typedef struct {
    int64_t NL, NG, nnz, nblocks;
    int32_t seg_max;
    int32_t reserved;
    const int32_t *scatterIds;
    const int32_t *rowStarts;
    const int32_t *localIds;
    const int32_t *blockStarts;
    /* NULL: one-pass kernels (random 8-byte accesses to HBM).  Else the
     * two-pass tiled kernels of the plan (all HBM accesses in runs). */
    const bs_plan_dev *plan;
} bs_gs_dev;

/* ---- errors -------------------------------------------------------------- */
const char *bs_strerror(int status);
/* Last error message recorded on `ctx` (empty string if none). */
const char *bs_last_error(const bs_ctx *ctx);

/* ---- context ------------------------------------------------------------- */
/* Creates a context on CUDA device `device`: queries its SM count and L2
 * size and allocates the reduction workspace (per-block partial sums, a
 * completion counter, a device error flag), about 64 KB.  *out is owned by
 * the caller and released by bs_ctx_destroy. */
int bs_ctx_create(int device, bs_ctx **out);
int bs_ctx_destroy(bs_ctx *ctx);
/* Number of SMs of the context's device. */
int bs_ctx_num_sms(const bs_ctx *ctx);
/* Synchronises `stream`, then reads and clears the device error flag that
 * the gather/scatter kernels raise on an out-of-range table entry (they
 * skip that entry instead of touching memory out of bounds) and that
 * bs_cg_solve_fused raises when a grid barrier gives up waiting.
 * *out_status is BS_OK, BS_EBOUNDS or BS_ETIMEOUT. */
int bs_ctx_device_status(bs_ctx *ctx, void *stream, int *out_status);

/* ---- BS1-BS5: mesh-free vector operations ---------------------------------
 * "Portable high-order finite element kernels I: Streaming Operations":
 * Benchmark Streaming test list and the CG vector operations (vector
 * addition y = alpha x + beta y, dot product alpha = x.y, norm alpha = x.x).
 */

/* BS1 copy: y[i] = x[i], i < n.  x == y is allowed; other overlap is not. */
int bs_copy(bs_ctx *ctx, int64_t n, const double *x, double *y, void *stream);

/* BS2 AXPY: y[i] = fma(alpha, x[i], beta * y[i]) with beta * y[i] rounded
 * first (for beta == 1 that product is exact and omitted).  x == y allowed. */
int bs_axpy(bs_ctx *ctx, int64_t n, double alpha, const double *x, double beta, double *y,
            void *stream);

/* BS2 with beta formed on the device: beta = *beta_num_dev / *beta_den_dev
 * (0 where the denominator is 0), then as bs_axpy.  CG's direction update
 * p = r + beta p with beta = rr_new / rr (alpha = 1) without a host round
 * trip.  The scalars must not lie inside y. */
int bs_axpy_dev(bs_ctx *ctx, int64_t n, double alpha, const double *x,
                const double *beta_num_dev, const double *beta_den_dev, double *y,
                void *stream);

/* BS3 norm: *out_dev = sum_i x[i]^2 -- the squared 2-norm, "norm:
 * alpha = x.x"; take the square root yourself. */
int bs_norm(bs_ctx *ctx, int64_t n, const double *x, double *out_dev, void *stream);

/* BS4 inner product: *out_dev = sum_i x[i] y[i]. */
int bs_dot(bs_ctx *ctx, int64_t n, const double *x, const double *y, double *out_dev,
           void *stream);

/* BS5 fused CG update (CG steps 8-10 fused into one pass):
 *   x[i] = fma(alpha, p[i], x[i]);  r[i] = fma(-alpha, Ap[i], r[i]);
 *   *rdotr_dev = sum_i r[i]^2 over the updated r.
 * alpha is `alpha` unless both alpha_num_dev and alpha_den_dev are given,
 * in which case alpha = *alpha_num_dev / *alpha_den_dev is formed on the
 * device (CG's alpha = (r.r) / (p.Ap) without a host round trip); a zero
 * denominator gives alpha = 0 (p = 0 only at an exact solution).
 * rdotr_dev may be NULL (no reduction).  x and r must not overlap each
 * other or p, Ap. */
int bs_cg_update(bs_ctx *ctx, int64_t n, const double *alpha_num_dev,
                 const double *alpha_den_dev, double alpha, const double *p, const double *Ap,
                 double *x, double *r, double *rdotr_dev, void *stream);

/* ---- mesh and index tables (host) -----------------------------------------
 * A box of E x E x E hexahedra of degree N on [0,1]^3 ("Portable high-order
 * finite element kernels I", eq. (1): K hexahedra, (p+1)^3 GLL nodes each,
 * N_L = K (p+1)^3).  Lattice element (ex,ey,ez) is number ex + E(ey + E ez);
 * storage slot s holds lattice element elemPerm[s]; local node (i,j,k) of
 * slot s has local index s (N+1)^3 + i + (N+1)(j + (N+1)k) and lies on
 * lattice node (ex N + w0, ey N + w1, ez N + w2), numbered x fastest on the
 * (EN+1)^3 lattice, with w = (i, j, k) rotated by the element's orientation
 * (identity unless ROTATE_ELEMS); its global id is nodePerm[lattice number].
 * Permutations (flags SHUFFLE_ELEMS / PERMUTE_GLOBAL, else identity): the
 * indices 0..n-1 ordered by (z_i, i), z_i the i-th SplitMix64 output from
 * state seed XOR (tag * 0x9E3779B97F4A7C15), tag 1 for elements, 2 for
 * global nodes.  Orientations (ROTATE_ELEMS): lattice element e takes
 * rotation ((z_e >> 11) * 24) >> 53 of stream tag 10, an index into the 24
 * proper rotations of the cube ordered by axis permutation (lexicographic:
 * output axis a takes input axis perm[a]) and then flip mask f = 0..7 (bit
 * a reverses output axis a, w_a = N - v[perm[a]]), keeping determinant +1;
 * rotation 0 is the identity.  MASK_BOUNDARY masks the local nodes on the
 * box boundary (-1), rotated or not.
 * Tables: scatterIds (local -> global, "scatterIds", negative = masked),
 * the CSR of Z^T with rows in global-id order and each row's local ids
 * ascending, and blockStarts grouping consecutive rows into segments of at
 * most seg_target CSR entries (the pages' blockStarts / NODES_PER_BLOCK).
 * Setup cost only; never timed. */
int bs_mesh_build_box(int E, int N, uint64_t seed, uint32_t flags, bs_mesh **out);
/* Same with an explicit segment target, 1 <= seg_target <= BS_GATHER_SEG_MAX
 * and seg_target >= 8 (the largest row). */
int bs_mesh_build_box_ex(int E, int N, uint64_t seed, uint32_t flags, int32_t seg_target,
                         bs_mesh **out);
/* The same tables (CSR of Z^T, row segments, default two-pass plan) for any
 * mesh, from the caller's local-to-global table: scatterIds[NL] (host,
 * copied) with every entry in [-1, NG), -1 = masked local ("GPU accelerated
 * spectral finite elements on all-hex meshes": I_{l->g}; any element shapes,
 * orientations and numbering).  Rows (the local copies of a global node) may
 * have up to BS_GATHER_SEG_MAX entries; the two-pass plan needs at most 32
 * (else it is left invalid and the one-pass kernels serve).  8 <= seg_target
 * <= BS_GATHER_SEG_MAX.  The mesh info reports E = N = K = 0, flags = 0.
 * BS_EBOUNDS for an entry outside [-1, NG), BS_EINVAL for bad sizes or a row
 * longer than BS_GATHER_SEG_MAX. */
int bs_mesh_from_ids(int64_t NL, int64_t NG, const int32_t *scatterIds, int32_t seg_target,
                     bs_mesh **out);
int bs_mesh_info(const bs_mesh *mesh, bs_mesh_info_t *out);
/* Host views of the four tables, owned by the mesh (valid until destroy).
 * Any output pointer may be NULL. */
int bs_mesh_tables(const bs_mesh *mesh, const int32_t **scatterIds, const int32_t **rowStarts,
                   const int32_t **localIds, const int32_t **blockStarts);
/* Checks every table invariant (ranges, CSR consistency with scatterIds,
 * ascending rows, segment sizes).  BS_OK, BS_EBOUNDS or BS_EINVAL. */
int bs_mesh_validate(const bs_mesh *mesh);
int bs_mesh_destroy(bs_mesh *mesh);

/* Two-pass gather/scatter plan, built with every mesh (default sizes) and
 * rebuilt by bs_mesh_plan with other sizes.  It reorders the data movement
 * only: the results are bitwise those of the one-pass kernels.
 *   Scatter: tiles of consecutive global rows (their q_G values staged in
 *   shared memory) write, per bucket of consecutive locals, one contiguous
 *   run of the work array (pass 1); each bucket then places its runs by
 *   local offset in shared memory and writes its q_L range coalesced
 *   (pass 2).
 *   Gather: tiles of consecutive locals write per-bucket runs, a bucket
 *   being `cluster` consecutive sub-buckets of rows with at most
 *   g_bucket_entries entries and rows each (pass 1); each bucket places its
 *   values in shared memory grouped by row length (each group an
 *   entries x rows column-major block), sums every row in ascending local
 *   order and writes its rows of q_G in order (pass 2).
 *   Rows may have at most 32 entries (box meshes: 8).
 * A tile or bucket is held by a cluster of `cluster` (1, 2 or 4) thread
 * blocks sharing their shared memory; the sizes are per block: a scatter
 * tile has cluster * s_tile_rows rows, and so on.  cluster * size must be
 * <= 32768 for the tiles (s_tile_rows, g_tile_len: pass-1 offsets are 15
 * bits, bit 15 marking the first slot of each run), <= 65536 for
 * s_bucket_len and <= 65535 for g_bucket_entries (>= 8).  A plan whose
 * kernels would need more than 227 KB of shared memory per block is left
 * invalid (valid = 0); then use the one-pass kernels. */
typedef struct {
    int32_t valid, cluster;
    int32_t s_tile_rows, s_bucket_len, g_tile_len, g_bucket_entries;
    int32_t s_ntiles, s_nbuckets, g_ntiles, g_nbuckets;
    int32_t g_bucket_rows_max, g_bucket_entries_max;
    int32_t g_mmax, reserved;                   /* longest row (<= 32) */
    int64_t smem_s1, smem_s2, smem_g1, smem_g2; /* bytes per block */
} bs_plan_info_t;
int bs_mesh_plan(bs_mesh *mesh, int32_t s_tile_rows, int32_t s_bucket_len, int32_t g_tile_len,
                 int32_t g_bucket_entries, int32_t cluster);
int bs_mesh_plan_info(const bs_mesh *mesh, bs_plan_info_t *out);
/* Host views of the plan's tables (owned by the mesh); any output may be
 * NULL.  BS_EINVAL if the plan is invalid. */
int bs_mesh_plan_tables(const bs_mesh *mesh, const int32_t **s_tileRows,
                        const int32_t **s_runStart, const uint16_t **s_src, const uint16_t **s_dst,
                        const int32_t **g_subRows, const int32_t **g_tileSlot,
                        const int32_t **g_runStart, const uint16_t **g_src,
                        const uint16_t **g_pos, const uint16_t **g_groupStart,
                        const uint16_t **g_rowPos);

/* ---- BS6 / BS7 -----------------------------------------------------------
 * "Portable high-order finite element kernels I": the BS6 gather kernel
 * (CSR of Z^T without values, rows blocked by blockStarts, entries staged
 * in shared memory) and the BS7 scatter kernel (scatterIds, negative =
 * masked); "GPU accelerated spectral finite elements on all-hex meshes":
 * local-to-global and global-to-local tables.
 * qL and qG must not overlap (BS_EINVAL).  Table entries out of range are
 * skipped and raise the device error flag (see bs_ctx_device_status). */

/* BS6 gather: qG[g] = (+0.0 + qL[l1]) + qL[l2] + ..., l1 < l2 < ... the
 * local copies of global node g; a row with no entries gives +0.0.
 * With t->plan the two-pass kernels run, except that a q_L of at most 8 MB
 * (BS7: a q_G of at most 32 MB) takes the one-pass kernels, faster for
 * vectors that stay in L2 (same results; BS_TUNE_ONEPASS=0 in the
 * environment at context creation turns this off). */
int bs_gather(bs_ctx *ctx, const bs_gs_dev *t, const double *qL, double *qG, void *stream);

/* BS7 scatter: qL[l] = qG[scatterIds[l]], or +0.0 where scatterIds[l] < 0. */
int bs_scatter(bs_ctx *ctx, const bs_gs_dev *t, const double *qG, double *qL, void *stream);

/* ---- global operator of a diagonal element-local operator ------------------
 * "Portable high-order finite element kernels I", eqs. (6)-(7): the global
 * operators are S_G = Z^T S_L Z and M_G = Z^T M_L Z with block-diagonal local
 * operators.  For a diagonal M_L with entries dL[l] (a lumped or GLL mass
 * matrix) this computes
 *   yG = Z^T (dL .* (Z xG)),  yG[g] = sum over l in row g, ascending, of
 *   (dL[l] * xG[g]) rounded, starting from +0.0 --
 * bitwise equal to bs_scatter, an elementwise product, and bs_gather.
 * Fused: scatter pass 1, then one kernel that places the scatter runs of a
 * local range, scales them and emits the gather runs of the same range, then
 * gather pass 2 -- q_L never reaches HBM.  Needs t->plan with cluster 1,
 * s_bucket_len == g_tile_len (the default plan) and work_len >= 2 nnz.
 * xG [NG], dL [NL], yG [NG] device; yG must not overlap xG or dL.
 * dL == NULL is the identity local operator: yG = Z^T Z xG (each global
 * value times its number of local copies, summed as the gather sums). */
int bs_apply_diag(bs_ctx *ctx, const bs_gs_dev *t, const double *xG, const double *dL,
                  double *yG, void *stream);

/* ---- one CG iteration's streaming sequence --------------------------------
 * With the identity as the element-local operator (S_G = Z^T S_L Z of eqs.
 * (6)-(7) with S_L = I): pL = Z pG (BS7); ApG = Z^T pL (BS6);
 * *pAp_dev = pG.ApG (BS4); alpha = *rr_dev / *pAp_dev;
 * xG += alpha pG, rG -= alpha ApG, *rr_new_dev = rG.rG (BS5);
 * *rnorm_dev = rG.rG (BS3).  pL is caller scratch of length t->NL; the
 * other vectors have length t->NG.  Five launches on `stream`. */
int bs_cg_iteration(bs_ctx *ctx, const bs_gs_dev *t, const double *pG, double *pL, double *ApG,
                    double *xG, double *rG, const double *rr_dev, double *pAp_dev,
                    double *rr_new_dev, double *rnorm_dev, void *stream);

/* ---- conjugate gradients on the global operator --------------------------
 * "Portable high-order finite element kernels I": every benchmark problem
 * solves its system by CG (its Algorithm 1, whose vector operations are
 * y = alpha x + beta y, dot, norm and y = A x, with steps 8-10 fusable into
 * BS5).  The algorithm's listing did not survive; this is the textbook
 * (Hestenes-Stiefel) iteration those operations and that fusion describe,
 * on A = Z^T diag(dL) Z (bs_apply_diag; dL == NULL: A = Z^T Z):
 *   ApG = A xG;  rG = bG - ApG  (copy, then BS2 with alpha = -1);
 *   pG = rG;  rr_0 = rG.rG (BS3)
 *   for k = 0 .. iters-1:
 *     ApG = A pG;  pAp_k = pG.ApG (BS4);  alpha = rr_k / pAp_k;
 *     xG += alpha pG, rG -= alpha ApG, rr_{k+1} = rG.rG (BS5);
 *     pG = rG + (rr_{k+1} / rr_k) pG (bs_axpy_dev)
 * A zero denominator makes its quotient 0 (exact convergence keeps x).
 * Every scalar stays on the device: scal_dev [2 iters + 1] receives
 * rr_0 .. rr_iters, then pAp_0 .. pAp_{iters-1}.  xG holds x_0 on entry
 * and x_iters on return; rG, pG, ApG [NG] are caller scratch (r_iters and
 * p_iters on return).  Needs a plan as bs_apply_diag does.  Launches
 * 3 + 4 + 6 iters kernels on `stream` and never synchronises, so the whole
 * solve can be captured in a CUDA graph.  No convergence test: the caller
 * reads rr_k when it chooses. */
int bs_cg_solve(bs_ctx *ctx, const bs_gs_dev *t, const double *dL, const double *bG, double *xG,
                double *rG, double *pG, double *ApG, int32_t iters, double *scal_dev,
                void *stream);

/* The same iteration as bs_cg_solve (same operations, same order of
 * arithmetic for every vector entry; the reductions sum in another order)
 * in ONE cooperative kernel: every block stays resident and the blocks
 * meet at grid barriers (four per iteration: after the scatter with the
 * local operator, after the CSR gather with p.Ap summed in the same pass,
 * after BS5, after the p update), so an iteration costs no launch at all.
 * For meshes small enough that launches set the time (the one-pass
 * gather/scatter phases do random 8-byte accesses); no plan is needed.
 * pL [NL] is caller scratch (q_L).  Each barrier wait is bounded: if one
 * gives up, the kernel ends early and bs_ctx_device_status reports
 * BS_ETIMEOUT.  Uses the context's reduction workspace (one call at a time
 * per context).  BS_ECUDA if the device cannot run the grid cooperatively. */
int bs_cg_solve_fused(bs_ctx *ctx, const bs_gs_dev *t, const double *dL, const double *bG,
                      double *xG, double *rG, double *pG, double *ApG, double *pL, int32_t iters,
                      double *scal_dev, void *stream);

/* Diagnostic of bs_cg_solve_fused's grid barrier: a cooperative grid of one
 * block per SM meets twice at the barrier.  With absent_block < 0 every
 * block arrives (bs_ctx_device_status then reports BS_OK); with
 * absent_block = b, block b leaves without arriving and every other block's
 * bounded wait runs out (~0.1-0.5 s): the kernel ends and
 * bs_ctx_device_status reports BS_ETIMEOUT.  Nothing faults or hangs. */
int bs_probe_grid_barrier(bs_ctx *ctx, int absent_block, void *stream);

/* ---- allocation-free inner product ----------------------------------------
 * The paper has no counterpart to this entry point; it is a library
 * convenience.  For callers that cannot call cudaMalloc -- code running
 * inside a device-memory allocator's own hooks, where an allocation would
 * recurse into the allocator, or an embedding runtime that owns every
 * device allocation -- and therefore cannot create a bs_ctx (a context
 * allocates its reduction workspace).
 *
 * Computes *out_dev = sum_i x[i] y[i] like bs_dot, with the same kernel,
 * but keeps the per-block partial sums and the completion counter in one
 * static device array of 8,448 bytes (1,024 partial sums plus the
 * counter) that every GPU loading this library holds until the process
 * exits.  It calls no cudaMalloc, cudaFree or allocating library routine.
 *  - Uses the calling thread's current device; x, y and out_dev must be
 *    memory of that device.  Every call looks up the array's device address
 *    (cudaGetSymbolAddress) and the SM count, so it stays valid across
 *    cudaDeviceReset.  The first call in a process may load the library's
 *    device code (lazy module loading); make it before any stream capture.
 *  - Do not call it from inside a CUDA host function or stream callback:
 *    CUDA forbids CUDA API calls there, and this call issues a memset and a
 *    kernel launch.
 *  - Each call first clears the counter on `stream` (the array keeps the
 *    previous call's contents).  All calls share the one array, so calls
 *    whose work overlaps on the GPU (other streams, other threads) race and
 *    give wrong results: serialise them.
 *  - BS_EINVAL if the device would need more than 1,024 partial sums
 *    (more than 256 SMs) or on a bad argument; BS_ECUDA on a CUDA error.
 *    If a CUDA error is already pending on the calling thread (left by
 *    earlier work), the call returns BS_ECUDA, launches nothing and leaves
 *    that error pending for its owner.  There is no context, so there is
 *    no error message beyond the code. */
int bs_dot_noalloc(int64_t n, const double *x, const double *y, double *out_dev, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* BS_H */
