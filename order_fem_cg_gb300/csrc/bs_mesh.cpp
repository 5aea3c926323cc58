// bs_mesh.cpp -- box hex mesh and its gather/scatter index tables (host).
//
// "Portable high-order finite element kernels I: Streaming Operations":
// K hexahedra with (p+1)^3 GLL nodes each (eq. (1)), the local vector of
// length N_L = K (p+1)^3 ordered by element, the scatter operator Z of
// eq. (3) stored as scatterIds (negative = masked), and the gather operator
// Z^T stored as CSR without values plus blockStarts, rows grouped so each
// thread block reads about NODES_PER_BLOCK entries.  "GPU accelerated
// spectral finite elements on all-hex meshes": these are the tables
// I_{l->g} and I_{g->l}.
//
// Numbering (setup convention of this library, stated in bs.h): lattice
// element ex + E(ey + E ez); slot s holds lattice element elemPerm[s];
// local index s (N+1)^3 + i + (N+1)(j + (N+1)k); lattice node
// (ex N + w0, ey N + w1, ez N + w2), x fastest, where w is (i, j, k) under
// the element's rotation (the identity unless BS_MESH_ROTATE_ELEMS); global
// id nodePerm[lattice].  Seeded permutations: indices ordered by
// (SplitMix64 draw, index); rotations: ((draw >> 11) * 24) >> 53.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <new>
#include <thread>
#include <vector>

#include "bs_mesh_impl.h"

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

inline uint64_t splitmix_out(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

template <class F>
void parallel_for(int64_t n, F &&f)
{
    unsigned hw = std::thread::hardware_concurrency();
    int64_t nt = hw ? static_cast<int64_t>(hw) : 1;
    if (nt > 32)
        nt = 32;
    if (n < (1 << 16) || nt == 1) {
        f(int64_t(0), n);
        return;
    }
    std::vector<std::thread> th;
    for (int64_t k = 0; k < nt; ++k) {
        int64_t a = n * k / nt, b = n * (k + 1) / nt;
        th.emplace_back([&f, a, b] { f(a, b); });
    }
    for (auto &t : th)
        t.join();
}

// Indices 0..n-1 ordered by (draw_i, i): a stable LSD radix sort on the
// 64-bit draws of stream (seed, tag), 8 passes of 8 bits.
std::vector<int32_t> seeded_permutation(uint64_t seed, uint64_t tag, int64_t n)
{
    const uint64_t state0 = seed ^ (tag * kGamma);
    std::vector<uint64_t> key(n), key2(n);
    std::vector<int32_t> idx(n), idx2(n);
    parallel_for(n, [&](int64_t a, int64_t b) {
        for (int64_t i = a; i < b; ++i) {
            key[i] = splitmix_out(state0 + static_cast<uint64_t>(i + 1) * kGamma);
            idx[i] = static_cast<int32_t>(i);
        }
    });
    for (int pass = 0; pass < 8; ++pass) {
        const int sh = 8 * pass;
        int64_t count[257] = {0};
        for (int64_t i = 0; i < n; ++i)
            ++count[((key[i] >> sh) & 255u) + 1];
        for (int d = 0; d < 256; ++d)
            count[d + 1] += count[d];
        for (int64_t i = 0; i < n; ++i) {
            const int64_t dst = count[(key[i] >> sh) & 255u]++;
            key2[dst] = key[i];
            idx2[dst] = idx[i];
        }
        key.swap(key2);
        idx.swap(idx2);
    }
    return idx;
}

// Rotation o of the reference cube as a signed axis permutation: output
// axis a takes input axis perm[a], reversed if flip[a].  The 24 proper
// rotations in the library's fixed order: permutations of (0, 1, 2) in
// lexicographic order, each with the flip masks 0..7 (bit a = axis a)
// whose matrix has determinant +1; rotation 0 is the identity.
struct Rotation {
    int perm[3];
    bool flip[3];
};

std::vector<Rotation> cube_rotations()
{
    std::vector<Rotation> r;
    int p[3] = {0, 1, 2};
    do {
        // parity of the permutation: count inversions
        const int inv = (p[0] > p[1]) + (p[0] > p[2]) + (p[1] > p[2]);
        for (int f = 0; f < 8; ++f) {
            const int nflip = (f & 1) + ((f >> 1) & 1) + ((f >> 2) & 1);
            if (((inv + nflip) & 1) != 0)
                continue;
            Rotation q;
            for (int a = 0; a < 3; ++a) {
                q.perm[a] = p[a];
                q.flip[a] = ((f >> a) & 1) != 0;
            }
            r.push_back(q);
        }
    } while (std::next_permutation(p, p + 3));
    return r;
}

// Rotation index in [0, 24) of every lattice element, from stream
// (seed, 10): ((draw >> 11) * 24) >> 53.
std::vector<uint8_t> seeded_orientations(uint64_t seed, int64_t K)
{
    const uint64_t state0 = seed ^ (10ull * kGamma);
    std::vector<uint8_t> o(K);
    parallel_for(K, [&](int64_t a, int64_t b) {
        for (int64_t e = a; e < b; ++e) {
            const uint64_t z = splitmix_out(state0 + static_cast<uint64_t>(e + 1) * kGamma);
            o[e] = static_cast<uint8_t>(((z >> 11) * 24u) >> 53);
        }
    });
    return o;
}

std::vector<int32_t> identity(int64_t n)
{
    std::vector<int32_t> v(n);
    for (int64_t i = 0; i < n; ++i)
        v[i] = static_cast<int32_t>(i);
    return v;
}

// From m->scatterIds (N_L entries in [-1, N_G)): the CSR of Z^T (rows in
// global-id order, local ids ascending per row), the row segments and the
// default two-pass plan.  Throws std::bad_alloc.
void finish_tables(bs_mesh *m)
{
    const int64_t NL = m->NL, NG = m->NG;
    const int64_t seg_target = m->seg_target;
    const int32_t *ids = m->scatterIds.data();
    m->rowStarts.assign(NG + 1, 0);
    int32_t *rs = m->rowStarts.data();
    for (int64_t l = 0; l < NL; ++l)
        if (ids[l] >= 0)
            ++rs[ids[l] + 1];
    int32_t max_row = 0;
    for (int64_t g = 0; g < NG; ++g) {
        max_row = std::max(max_row, rs[g + 1]);
        rs[g + 1] += rs[g];
    }
    m->max_row = max_row;
    m->nnz = rs[NG];
    m->localIds.resize(m->nnz);
    {
        std::vector<int32_t> pos(rs, rs + NG);
        for (int64_t l = 0; l < NL; ++l)
            if (ids[l] >= 0)
                m->localIds[pos[ids[l]]++] = static_cast<int32_t>(l);
    }

    // Row segments: consecutive rows, at most seg_target entries and at
    // most seg_target rows each.  seg_max = the largest of any segment's
    // entry and row counts: the shared-memory staging capacity needed.
    m->blockStarts.clear();
    m->blockStarts.push_back(0);
    int64_t ce = 0, cr = 0;
    int32_t seg_max = 0;
    for (int64_t g = 0; g < NG; ++g) {
        const int64_t len = rs[g + 1] - rs[g];
        if (cr > 0 && (ce + len > seg_target || cr + 1 > seg_target)) {
            m->blockStarts.push_back(static_cast<int32_t>(g));
            seg_max = std::max<int32_t>(seg_max, static_cast<int32_t>(std::max(ce, cr)));
            ce = 0;
            cr = 0;
        }
        ce += len;
        cr += 1;
    }
    seg_max = std::max<int32_t>(seg_max, static_cast<int32_t>(std::max(ce, cr)));
    m->blockStarts.push_back(static_cast<int32_t>(NG));
    m->seg_max = std::max<int32_t>(seg_max, 1);
    bs_plan_build(m, BS_TILE_S_ROWS, BS_TILE_S_BUCKET, BS_TILE_G_LOCALS, BS_TILE_G_BUCKET,
                  BS_TILE_CLUSTER);
}

// BS_FAULT=badtable: one out-of-range entry in each of scatterIds and
// localIds (the plan, built before, stays consistent).
void inject_bad_table(bs_mesh *m)
{
    if (!bs_fault("badtable"))
        return;
    if (m->NL > 0)
        m->scatterIds[m->NL / 2] = static_cast<int32_t>(m->NG);
    if (m->nnz > 0)
        m->localIds[m->nnz / 2] = static_cast<int32_t>(m->NL);
}

} // namespace

extern "C" int bs_mesh_build_box_ex(int E, int N, uint64_t seed, uint32_t flags,
                                    int32_t seg_target, bs_mesh **out)
{
    if (!out)
        return BS_EINVAL;
    *out = nullptr;
    if (E < 1 || N < 1 || seg_target < 8 || seg_target > BS_GATHER_SEG_MAX ||
        (flags & ~15u) != 0)
        return BS_EINVAL;
    const int64_t q = N + 1, Np = q * q * q, M = static_cast<int64_t>(E) * N + 1;
    const int64_t K = static_cast<int64_t>(E) * E * E;
    const int64_t NL = K * Np, NG = M * M * M;
    if (NL > INT32_MAX || NG >= INT32_MAX)
        return BS_EINVAL;

    bs_mesh *m = new (std::nothrow) bs_mesh();
    if (!m)
        return BS_ENOMEM;
    try {
        m->E = E;
        m->N = N;
        m->flags = flags;
        m->seg_target = seg_target;
        m->K = K;
        m->NL = NL;
        m->NG = NG;

        const std::vector<int32_t> elemPerm =
            (flags & BS_MESH_SHUFFLE_ELEMS) ? seeded_permutation(seed, 1, K) : identity(K);
        const std::vector<int32_t> nodePerm =
            (flags & BS_MESH_PERMUTE_GLOBAL) ? seeded_permutation(seed, 2, NG) : identity(NG);
        const bool mask = (flags & BS_MESH_MASK_BOUNDARY) != 0;
        const bool rotate = (flags & BS_MESH_ROTATE_ELEMS) != 0;
        const std::vector<uint8_t> orient =
            rotate ? seeded_orientations(seed, K) : std::vector<uint8_t>();
        const std::vector<Rotation> rot = cube_rotations();
        const int nrot = rotate ? 24 : 1;

        // Per rotation: the lattice offset of each element-local node from
        // the element's lattice corner, and its lattice coordinates in the
        // element (for the boundary mask).
        std::vector<int64_t> off(nrot * Np);
        std::vector<int32_t> ni(nrot * Np), nj(nrot * Np), nk(nrot * Np);
        for (int o = 0; o < nrot; ++o)
            for (int64_t k = 0, n = 0; k < q; ++k)
                for (int64_t j = 0; j < q; ++j)
                    for (int64_t i = 0; i < q; ++i, ++n) {
                        const int64_t v[3] = {i, j, k};
                        int64_t w[3];
                        for (int a = 0; a < 3; ++a) {
                            const int64_t c = v[rot[o].perm[a]];
                            w[a] = rot[o].flip[a] ? N - c : c;
                        }
                        off[o * Np + n] = w[0] + M * (w[1] + M * w[2]);
                        ni[o * Np + n] = static_cast<int32_t>(w[0]);
                        nj[o * Np + n] = static_cast<int32_t>(w[1]);
                        nk[o * Np + n] = static_cast<int32_t>(w[2]);
                    }

        m->scatterIds.resize(NL);
        int32_t *ids = m->scatterIds.data();
        parallel_for(K, [&](int64_t a, int64_t b) {
            for (int64_t s = a; s < b; ++s) {
                const int64_t e = elemPerm[s];
                const int64_t ex = e % E, ey = (e / E) % E, ez = e / (static_cast<int64_t>(E) * E);
                const int64_t base = ex * N + M * (ey * N + M * (ez * N));
                const int64_t ro = rotate ? orient[e] * Np : 0;
                int32_t *row = ids + s * Np;
                for (int64_t n = 0; n < Np; ++n) {
                    int32_t g = nodePerm[base + off[ro + n]];
                    if (mask) {
                        const int64_t gx = ex * N + ni[ro + n], gy = ey * N + nj[ro + n],
                                      gz = ez * N + nk[ro + n];
                        if (gx == 0 || gy == 0 || gz == 0 || gx == M - 1 || gy == M - 1 ||
                            gz == M - 1)
                            g = -1;
                    }
                    row[n] = g;
                }
            }
        });

        finish_tables(m);
    } catch (const std::bad_alloc &) {
        delete m;
        return BS_ENOMEM;
    }
    inject_bad_table(m);
    *out = m;
    return BS_OK;
}

extern "C" int bs_mesh_build_box(int E, int N, uint64_t seed, uint32_t flags, bs_mesh **out)
{
    return bs_mesh_build_box_ex(E, N, seed, flags, BS_GATHER_SEG_DEFAULT, out);
}

extern "C" int bs_mesh_from_ids(int64_t NL, int64_t NG, const int32_t *scatterIds,
                                int32_t seg_target, bs_mesh **out)
{
    if (!out)
        return BS_EINVAL;
    *out = nullptr;
    if (NL < 0 || NG < 0 || NL > INT32_MAX || NG >= INT32_MAX || (NL > 0 && !scatterIds) ||
        seg_target < 8 || seg_target > BS_GATHER_SEG_MAX)
        return BS_EINVAL;
    // every entry in [-1, N_G) (-1 = masked local)
    for (int64_t l = 0; l < NL; ++l)
        if (scatterIds[l] < -1 || scatterIds[l] >= NG)
            return BS_EBOUNDS;
    bs_mesh *m = new (std::nothrow) bs_mesh();
    if (!m)
        return BS_ENOMEM;
    try {
        m->seg_target = seg_target;
        m->NL = NL;
        m->NG = NG;
        m->scatterIds.assign(scatterIds, scatterIds + NL);
        finish_tables(m);
    } catch (const std::bad_alloc &) {
        delete m;
        return BS_ENOMEM;
    }
    if (m->seg_max > BS_GATHER_SEG_MAX) {  // a row longer than the gather's staging
        delete m;
        return BS_EINVAL;
    }
    inject_bad_table(m);
    *out = m;
    return BS_OK;
}

extern "C" int bs_mesh_info(const bs_mesh *m, bs_mesh_info_t *out)
{
    if (!m || !out)
        return BS_EINVAL;
    out->E = m->E;
    out->N = m->N;
    out->flags = m->flags;
    out->max_row = m->max_row;
    out->K = m->K;
    out->NL = m->NL;
    out->NG = m->NG;
    out->nnz = m->nnz;
    out->nblocks = static_cast<int64_t>(m->blockStarts.size()) - 1;
    out->seg_max = m->seg_max;
    out->seg_target = m->seg_target;
    return BS_OK;
}

extern "C" int bs_mesh_tables(const bs_mesh *m, const int32_t **scatterIds,
                              const int32_t **rowStarts, const int32_t **localIds,
                              const int32_t **blockStarts)
{
    if (!m)
        return BS_EINVAL;
    if (scatterIds)
        *scatterIds = m->scatterIds.data();
    if (rowStarts)
        *rowStarts = m->rowStarts.data();
    if (localIds)
        *localIds = m->localIds.data();
    if (blockStarts)
        *blockStarts = m->blockStarts.data();
    return BS_OK;
}

extern "C" int bs_mesh_validate(const bs_mesh *m)
{
    if (!m)
        return BS_EINVAL;
    const int64_t NL = m->NL, NG = m->NG;
    if (static_cast<int64_t>(m->scatterIds.size()) != NL ||
        static_cast<int64_t>(m->rowStarts.size()) != NG + 1 ||
        static_cast<int64_t>(m->localIds.size()) != m->nnz || m->blockStarts.size() < 2)
        return BS_EINVAL;
    const int32_t *ids = m->scatterIds.data();
    const int32_t *rs = m->rowStarts.data();
    const int32_t *li = m->localIds.data();
    int64_t unmasked = 0;
    for (int64_t l = 0; l < NL; ++l) {
        if (ids[l] >= NG || ids[l] < -1)
            return BS_EBOUNDS;
        unmasked += ids[l] >= 0;
    }
    if (unmasked != m->nnz || rs[0] != 0 || rs[NG] != m->nnz)
        return BS_EBOUNDS;
    for (int64_t g = 0; g < NG; ++g) {
        if (rs[g + 1] < rs[g] || rs[g + 1] - rs[g] > m->max_row)
            return BS_EBOUNDS;
        for (int64_t e = rs[g]; e < rs[g + 1]; ++e) {
            const int32_t l = li[e];
            if (l < 0 || l >= NL || ids[l] != g)
                return BS_EBOUNDS;
            if (e > rs[g] && li[e - 1] >= l)
                return BS_EBOUNDS;
        }
    }
    // Each unmasked local appears exactly once: row membership is forced by
    // ids[l] == g and rows are strictly ascending, so counts suffice.
    const int32_t *bs = m->blockStarts.data();
    const int64_t nb = static_cast<int64_t>(m->blockStarts.size()) - 1;
    if (bs[0] != 0 || bs[nb] != NG)
        return BS_EBOUNDS;
    for (int64_t b = 0; b < nb; ++b) {
        if (bs[b + 1] <= bs[b] && NG > 0)
            return BS_EBOUNDS;
        const int64_t ne = rs[bs[b + 1]] - rs[bs[b]];
        if (ne > m->seg_max || bs[b + 1] - bs[b] > m->seg_max || m->seg_max > BS_GATHER_SEG_MAX)
            return BS_EBOUNDS;
    }
    return BS_OK;
}

extern "C" int bs_mesh_destroy(bs_mesh *m)
{
    delete m;
    return BS_OK;
}

extern "C" int bs_mesh_plan(bs_mesh *m, int32_t s_tile_rows, int32_t s_bucket_len,
                            int32_t g_tile_len, int32_t g_bucket_entries, int32_t cluster)
{
    if (!m)
        return BS_EINVAL;
    try {
        bs_plan_build(m, s_tile_rows, s_bucket_len, g_tile_len, g_bucket_entries, cluster);
    } catch (const std::bad_alloc &) {
        m->plan = bs_plan();
        return BS_ENOMEM;
    }
    return m->plan.valid ? BS_OK : BS_EINVAL;
}

extern "C" int bs_mesh_plan_info(const bs_mesh *m, bs_plan_info_t *out)
{
    if (!m || !out)
        return BS_EINVAL;
    const bs_plan &p = m->plan;
    std::memset(out, 0, sizeof(*out));
    out->valid = p.valid ? 1 : 0;
    out->cluster = p.cluster;
    out->s_tile_rows = p.s_tile_rows;
    out->s_bucket_len = p.s_bucket_len;
    out->g_tile_len = p.g_tile_len;
    out->g_bucket_entries = p.g_bucket_entries;
    out->s_ntiles = p.s_ntiles;
    out->s_nbuckets = p.s_nbuckets;
    out->g_ntiles = p.g_ntiles;
    out->g_nbuckets = p.g_nbuckets;
    out->g_bucket_rows_max = p.g_bucket_rows_max;
    out->g_bucket_entries_max = p.g_bucket_entries_max;
    out->g_mmax = p.g_mmax;
    if (p.valid) {
        out->smem_s1 = bs_plan_smem_s1(p);
        out->smem_s2 = bs_plan_smem_s2(p);
        out->smem_g1 = bs_plan_smem_g1(p);
        out->smem_g2 = bs_plan_smem_g2(p);
    }
    return BS_OK;
}

extern "C" int bs_mesh_plan_tables(const bs_mesh *m, const int32_t **s_tileRows,
                                   const int32_t **s_runStart, const uint16_t **s_src,
                                   const uint16_t **s_dst, const int32_t **g_subRows,
                                   const int32_t **g_tileSlot, const int32_t **g_runStart,
                                   const uint16_t **g_src, const uint16_t **g_pos,
                                   const uint16_t **g_groupStart, const uint16_t **g_rowPos)
{
    if (!m || !m->plan.valid)
        return BS_EINVAL;
    const bs_plan &p = m->plan;
    if (s_tileRows) *s_tileRows = p.s_tileRows.data();
    if (s_runStart) *s_runStart = p.s_runStart.data();
    if (s_src) *s_src = p.s_src.data();
    if (s_dst) *s_dst = p.s_dst.data();
    if (g_subRows) *g_subRows = p.g_subRows.data();
    if (g_tileSlot) *g_tileSlot = p.g_tileSlot.data();
    if (g_runStart) *g_runStart = p.g_runStart.data();
    if (g_src) *g_src = p.g_src.data();
    if (g_pos) *g_pos = p.g_pos.data();
    if (g_groupStart) *g_groupStart = p.g_groupStart.data();
    if (g_rowPos) *g_rowPos = p.g_rowPos.data();
    return BS_OK;
}
