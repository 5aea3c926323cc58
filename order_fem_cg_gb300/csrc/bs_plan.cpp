// bs_plan.cpp -- two-pass gather/scatter plan of a mesh (host, setup only).
//
// The plan turns the random permutation between the CSR (global) order and
// the local order into two passes whose global-memory accesses are all
// contiguous runs; the random part happens in shared memory.  See
// bs_mesh_impl.h for the layout and bs_gs2.cu for the kernels.
#include <algorithm>
#include <cstring>

#include "bs_mesh_impl.h"

// Pass 1 holds the tile, the packed run scan (8 bytes per bucket, plus the
// totals) and the work offset of every run (4 bytes per bucket).
int64_t bs_plan_smem_s1(const bs_plan &p)
{
    return 8ll * p.s_tile_rows + 8ll * (p.s_nbuckets + 1) + 4ll * p.s_nbuckets;
}

int64_t bs_plan_smem_s2(const bs_plan &p)
{
    return 8ll * p.s_bucket_len;
}

int64_t bs_plan_smem_g1(const bs_plan &p)
{
    return 8ll * p.g_tile_len + 8ll * (p.g_nbuckets + 1) + 4ll * p.g_nbuckets;
}

int64_t bs_plan_smem_g2(const bs_plan &p)
{
    // staged values, then the sub-bucket's group table
    return 8ll * p.g_bucket_entries_max + 4ll * (BS_PLAN_MMAX + 1);
}

void bs_plan_build(bs_mesh *m, int32_t TRc, int32_t BLc, int32_t TLc, int32_t EBc, int32_t CS)
{
    m->plan = bs_plan();
    bs_plan &p = m->plan;
    if (CS != 1 && CS != 2 && CS != 4)
        return;
    // offsets inside a bucket (whole cluster) are stored as 16 bits, those
    // inside a tile as 15 bits (bit 15 marks the first slot of a run)
    if (TRc < 1 || BLc < 1 || TLc < 1 || EBc < 8 || static_cast<int64_t>(TRc) * CS > 32768 ||
        static_cast<int64_t>(BLc) * CS > 65536 || static_cast<int64_t>(TLc) * CS > 32768 ||
        static_cast<int64_t>(EBc) * CS > 65535)
        return;
    const int64_t NL = m->NL, NG = m->NG, nnz = m->nnz;
    const int32_t *rs = m->rowStarts.data();
    const int32_t *li = m->localIds.data();
    const int32_t *ids = m->scatterIds.data();
    p.cluster = CS;
    p.s_tile_rows = TRc;
    p.s_bucket_len = BLc;
    p.g_tile_len = TLc;
    p.g_bucket_entries = EBc;
    const int64_t TR = static_cast<int64_t>(TRc) * CS, BL = static_cast<int64_t>(BLc) * CS;
    const int64_t TL = static_cast<int64_t>(TLc) * CS;

    // ------------------------------------------------------------ scatter
    const int64_t T = (NG + TR - 1) / TR, B = (NL + BL - 1) / BL;
    p.s_ntiles = static_cast<int32_t>(T);
    p.s_nbuckets = static_cast<int32_t>(B);
    if (bs_plan_smem_s1(p) > BS_SMEM_MAX || bs_plan_smem_s2(p) > BS_SMEM_MAX ||
        static_cast<double>(T + 1) * B > 2e9) {
        m->plan = bs_plan();
        return;
    }
    p.s_tileRows.resize(T + 1);
    for (int64_t t = 0; t <= T; ++t)
        p.s_tileRows[t] = static_cast<int32_t>(std::min<int64_t>(t * TR, NG));
    {
        std::vector<int32_t> cnt(static_cast<size_t>(T) * B, 0);
        for (int64_t t = 0; t < T; ++t)
            for (int64_t e = rs[p.s_tileRows[t]]; e < rs[p.s_tileRows[t + 1]]; ++e)
                ++cnt[t * B + li[e] / BL];
        // work order: bucket-major, then tile, then CSR order
        p.s_runStart.resize(static_cast<size_t>(T + 1) * B);
        int64_t pos = 0;
        for (int64_t b = 0; b < B; ++b) {
            for (int64_t t = 0; t < T; ++t) {
                p.s_runStart[t * B + b] = static_cast<int32_t>(pos);
                pos += cnt[t * B + b];
            }
            p.s_runStart[T * B + b] = static_cast<int32_t>(pos);
        }
        p.s_src.resize(nnz);
        p.s_dst.resize(nnz);
        std::vector<int32_t> off(B), cur(B);
        for (int64_t t = 0; t < T; ++t) {
            int32_t acc = 0;
            for (int64_t b = 0; b < B; ++b) {
                off[b] = acc;
                acc += cnt[t * B + b];
                cur[b] = 0;
            }
            const int32_t r0 = p.s_tileRows[t];
            const int64_t base = rs[r0];
            for (int32_t g = r0; g < p.s_tileRows[t + 1]; ++g)
                for (int64_t e = rs[g]; e < rs[g + 1]; ++e) {
                    const int32_t l = li[e];
                    const int64_t b = l / BL;
                    const int32_t k = cur[b]++;
                    p.s_src[base + off[b] + k] =
                        static_cast<uint16_t>((g - r0) | (k == 0 ? BS_PLAN_RUN_START : 0));
                    p.s_dst[p.s_runStart[t * B + b] + k] = static_cast<uint16_t>(l - b * BL);
                }
        }
    }

    // ------------------------------------------------------------- gather
    const int64_t U = (NL + TL - 1) / TL;
    p.g_ntiles = static_cast<int32_t>(U);
    // sub-buckets: consecutive rows, at most EBc entries and EBc rows each;
    // a bucket is CS consecutive sub-buckets (padded with empty ones)
    std::vector<int32_t> subOf(NG);
    p.g_subRows.clear();
    p.g_subRows.push_back(0);
    {
        int64_t ce = 0, cr = 0;
        int32_t emax = 0, rmax = 0;
        for (int64_t g = 0; g < NG; ++g) {
            const int64_t len = rs[g + 1] - rs[g];
            if (cr > 0 && (ce + len > EBc || cr + 1 > EBc)) {
                p.g_subRows.push_back(static_cast<int32_t>(g));
                emax = std::max<int32_t>(emax, static_cast<int32_t>(ce));
                rmax = std::max<int32_t>(rmax, static_cast<int32_t>(cr));
                ce = 0;
                cr = 0;
            }
            subOf[g] = static_cast<int32_t>(p.g_subRows.size()) - 1;
            ce += len;
            cr += 1;
        }
        emax = std::max<int32_t>(emax, static_cast<int32_t>(ce));
        rmax = std::max<int32_t>(rmax, static_cast<int32_t>(cr));
        p.g_subRows.push_back(static_cast<int32_t>(NG));
        while ((p.g_subRows.size() - 1) % CS != 0)
            p.g_subRows.push_back(static_cast<int32_t>(NG));
        p.g_bucket_entries_max = std::max<int32_t>(emax, 1);
        p.g_bucket_rows_max = std::max<int32_t>(rmax, 1);
    }
    const int64_t C = (static_cast<int64_t>(p.g_subRows.size()) - 1) / CS;
    p.g_nbuckets = static_cast<int32_t>(C);
    if (bs_plan_smem_g1(p) > BS_SMEM_MAX || bs_plan_smem_g2(p) > BS_SMEM_MAX ||
        static_cast<double>(U + 1) * C > 2e9) {
        m->plan = bs_plan();
        return;
    }
    // rows grouped by length inside each sub-bucket; the R rows of length m
    // of a group form an m x R column-major block: entry j of the group's
    // row q sits at groupStart[m-1] + j R + q, so that consecutive threads
    // summing consecutive rows read consecutive shared-memory words
    const int32_t MM = std::max<int32_t>(m->max_row, 1);
    if (MM > BS_PLAN_MMAX) {
        m->plan = bs_plan();
        return;
    }
    p.g_mmax = MM;
    const int64_t NS = static_cast<int64_t>(p.g_subRows.size()) - 1;
    p.g_groupStart.assign(static_cast<size_t>(NS) * (MM + 1), 0);
    p.g_rowPos.assign(NG, 0xFFFF);
    for (int64_t sb = 0; sb < NS; ++sb) {
        uint16_t *gs = p.g_groupStart.data() + sb * (MM + 1);
        int32_t cnt[BS_PLAN_MMAX + 1] = {0};
        for (int32_t g = p.g_subRows[sb]; g < p.g_subRows[sb + 1]; ++g)
            ++cnt[rs[g + 1] - rs[g]];
        int32_t acc = 0, next[BS_PLAN_MMAX + 1];
        for (int32_t len = 1; len <= MM; ++len) {
            gs[len - 1] = static_cast<uint16_t>(acc);
            next[len] = acc;
            acc += cnt[len] * len;
        }
        gs[MM] = static_cast<uint16_t>(acc);
        for (int32_t g = p.g_subRows[sb]; g < p.g_subRows[sb + 1]; ++g) {
            const int32_t len = rs[g + 1] - rs[g];
            if (len > 0)
                p.g_rowPos[g] = static_cast<uint16_t>(next[len]++);
        }
    }
    // staged position of CSR entry e (row g of length m, k-th entry) within
    // its bucket: offset of its sub-bucket in the bucket + position of the
    // row in its group block + k times the group's row count
    std::vector<int32_t> epos(NL, -1);
    for (int64_t e = 0; e < nnz; ++e)
        epos[li[e]] = static_cast<int32_t>(e);
    p.g_tileSlot.resize(U + 1);
    {
        int64_t acc = 0;
        for (int64_t u = 0; u < U; ++u) {
            p.g_tileSlot[u] = static_cast<int32_t>(acc);
            const int64_t l1 = std::min<int64_t>((u + 1) * TL, NL);
            for (int64_t l = u * TL; l < l1; ++l)
                acc += ids[l] >= 0;
        }
        p.g_tileSlot[U] = static_cast<int32_t>(acc);
    }
    {
        std::vector<int32_t> cnt(static_cast<size_t>(U) * C, 0);
        for (int64_t l = 0; l < NL; ++l)
            if (ids[l] >= 0)
                ++cnt[(l / TL) * C + subOf[ids[l]] / CS];
        // work order: bucket-major (a bucket's range is its CSR range), then
        // tile, then ascending local id
        p.g_runStart.resize(static_cast<size_t>(U + 1) * C);
        for (int64_t c = 0; c < C; ++c) {
            int64_t pos = rs[p.g_subRows[c * CS]];
            for (int64_t u = 0; u < U; ++u) {
                p.g_runStart[u * C + c] = static_cast<int32_t>(pos);
                pos += cnt[u * C + c];
            }
            p.g_runStart[U * C + c] = static_cast<int32_t>(pos);
        }
        p.g_src.resize(nnz);
        p.g_pos.resize(nnz);
        std::vector<int32_t> off(C), cur(C);
        for (int64_t u = 0; u < U; ++u) {
            int32_t acc = 0;
            for (int64_t c = 0; c < C; ++c) {
                off[c] = acc;
                acc += cnt[u * C + c];
                cur[c] = 0;
            }
            const int64_t l0 = u * TL, l1 = std::min<int64_t>(l0 + TL, NL);
            const int64_t base = p.g_tileSlot[u];
            for (int64_t l = l0; l < l1; ++l) {
                const int32_t g = ids[l];
                if (g < 0)
                    continue;
                const int64_t c = subOf[g] / CS;
                const int32_t k = cur[c]++;
                p.g_src[base + off[c] + k] =
                    static_cast<uint16_t>((l - l0) | (k == 0 ? BS_PLAN_RUN_START : 0));
                const int64_t sb = subOf[g];
                const int64_t in_bucket = rs[p.g_subRows[sb]] - rs[p.g_subRows[c * CS]];
                const int32_t len = rs[g + 1] - rs[g];
                const uint16_t *gs = p.g_groupStart.data() + sb * (MM + 1);
                const int64_t R = (gs[len] - gs[len - 1]) / len;
                p.g_pos[p.g_runStart[u * C + c] + k] = static_cast<uint16_t>(
                    in_bucket + p.g_rowPos[g] + (epos[l] - rs[g]) * R);
            }
        }
    }
    p.valid = true;
}
