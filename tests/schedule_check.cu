// Host-only checks of the tcgen05 GEMM's work schedules (schedule.cuh), run on
// the CPU by tests/test_schedule.py: for many launch shapes and SM counts,
//   * one-CTA schedule (whole tiles, last-wave halves, split K): every output
//     tile column and every K block is covered by exactly one unit; a split
//     tile's pieces come from the CTAs sk_cta_of names, at most kMaxPieces of
//     them, each in its own workspace slot; the launch fits its workspace;
//   * pair schedule: every pair tile's columns are covered exactly once, with
//     halves only in a short last wave.
// Prints a summary line; exit status 1 on any failure.
#include "schedule.cuh"

#include <cstdio>
#include <set>
#include <vector>

using namespace sq::sched;

static long long g_checked = 0, g_fail = 0;
#define CHECK(cond, ...)                                                   \
    do {                                                                   \
        if (!(cond)) {                                                     \
            if (g_fail < 20) {                                             \
                std::printf("FAIL line %d: ", __LINE__);                   \
                std::printf(__VA_ARGS__);                                  \
                std::printf("\n");                                         \
            }                                                              \
            ++g_fail;                                                      \
        }                                                                  \
    } while (0)

static void check_one_cta(long long M, long long N, long long K, int sms, bool split) {
    int grid = 0;
    const Schedule sc = plan_launch(M, N, K, sms, split, &grid);
    const int m_tiles = (int)((M + BM - 1) / BM), n_tiles = (int)((N + BN - 1) / BN);
    const int nkb = (int)((K + BK - 1) / BK);
    CHECK(grid >= 1 && grid <= sms, "grid %d for sms %d", grid, sms);
    // coverage[(tile m, 32-column slice, K block)]
    const int slices = n_tiles * (BN / 32);
    std::vector<unsigned char> cover((size_t)m_tiles * slices * nkb, 0);
    std::vector<std::set<int>> piece_ctas(sc.sk_tiles > 0 ? sc.sk_tiles : 1);
    int min_units = 1 << 30, max_units = 0;
    for (int c = 0; c < grid; ++c) {
        Cursor cu;
        cursor_init(sc, cu, c);
        Work w;
        int units = 0;
        std::set<int> slots;
        while (next_work(sc, cu, w, grid)) {
            ++units;
            CHECK(w.m0 % BM == 0 && w.n0 % 128 == 0 && (w.bn == BN || w.bn == BN / 2),
                  "unit shape m0 %d n0 %d bn %d", w.m0, w.n0, w.bn);
            CHECK(0 <= w.kb0 && w.kb0 < w.kb1 && w.kb1 <= nkb, "K range %d..%d of %d", w.kb0,
                  w.kb1, nkb);
            const int mt = w.m0 / BM;
            CHECK(mt < m_tiles && w.n0 / BN < n_tiles, "tile out of range");
            if (mt >= m_tiles || w.n0 / BN >= n_tiles) continue;
            for (int col = w.n0; col < w.n0 + w.bn; col += 32)
                for (int kb = w.kb0; kb < w.kb1; ++kb)
                    ++cover[((size_t)mt * slices + col / 32) * nkb + kb];
            if (w.skt >= 0) {
                CHECK(w.skt < sc.sk_tiles, "split tile %d of %d", w.skt, sc.sk_tiles);
                if (w.skt < sc.sk_tiles) piece_ctas[w.skt].insert(c);
                const long long tb = (long long)w.skt * nkb;
                const int e = sk_start(sc, c) >= tb ? 0 : 1;
                CHECK(slots.insert(e).second, "CTA %d uses slot %d twice", c, e);
            }
        }
        min_units = units < min_units ? units : min_units;
        max_units = units > max_units ? units : max_units;
    }
    for (size_t i = 0; i < cover.size(); ++i)
        CHECK(cover[i] == 1, "M %lld N %lld K %lld sms %d split %d: cell %zu covered %d times", M,
              N, K, sms, (int)split, i, cover[i]);
    if (sc.sk_tiles == 0)
        CHECK(max_units - min_units <= 1, "unbalanced: %d..%d units per CTA", min_units,
              max_units);
    for (int r = 0; r < sc.sk_tiles; ++r) {
        const long long tb = (long long)r * nkb;
        const int c0 = sk_cta_of(sc, tb), c1 = sk_cta_of(sc, tb + nkb - 1);
        const std::set<int> &p = piece_ctas[r];
        if (p.empty()) continue;  // the whole tile lies in one CTA's share
        CHECK((int)p.size() == c1 - c0 + 1 && *p.begin() == c0 && *p.rbegin() == c1,
              "tile %d: pieces from %zu CTAs, sk_cta_of says %d..%d", r, p.size(), c0, c1);
        CHECK((int)p.size() <= kMaxPieces, "tile %d split into %zu pieces", r, p.size());
    }
    if (sc.sk_tiles > 0) {
        CHECK(sc.sk_tiles <= sc.sk_cnt_tiles, "counter block too small");
        CHECK(sk_workspace_bytes(sc) > 0 && sk_counter_bytes(sc) % 256 == 0, "workspace layout");
        CHECK(nkb >= kMinSplitKb && sc.dp_tiles == 0, "split outside its rule");
    }
    ++g_checked;
}

static void check_pair(long long M, long long N, int clusters) {
    const int m_pairs = (int)((M + 2 * BM - 1) / (2 * BM)), n_tiles = (int)((N + BN - 1) / BN);
    // planned for every cluster that fits, run on no more clusters than items
    const PairSchedule sc = make_pair_schedule(m_pairs, n_tiles, clusters);
    const int used = sc.items < clusters ? sc.items : clusters;
    std::vector<unsigned char> cover((size_t)m_pairs * n_tiles * 2, 0);
    for (int cl = 0; cl < used; ++cl) {
        for (int i = cl; i < sc.items; i += used) {
            int m0, n0, bn;
            pair_item_at(sc, i, m0, n0, bn);
            CHECK(m0 % (2 * BM) == 0 && n0 % 128 == 0 && (bn == BN || bn == BN / 2),
                  "pair item m0 %d n0 %d bn %d", m0, n0, bn);
            const int mp = m0 / (2 * BM);
            CHECK(mp < m_pairs && n0 / BN < n_tiles, "pair item out of range");
            if (mp >= m_pairs || n0 / BN >= n_tiles) continue;
            for (int col = n0; col < n0 + bn; col += 128) ++cover[((size_t)mp * n_tiles) * 2 + col / 128];
            if (bn < BN) CHECK(i >= sc.full_items, "half item outside the last wave");
        }
    }
    for (size_t i = 0; i < cover.size(); ++i)
        CHECK(cover[i] == 1, "pair M %lld N %lld clusters %d: half-tile %zu covered %d times", M,
              N, clusters, i, cover[i]);
    ++g_checked;
}

// The static scratch of sq_linear_i8_static_ws (SQ_STATIC_WORKSPACE_BYTES,
// 40 MiB) holds the split-K workspace of every shape on a GPU of up to 159 SMs;
// on larger GPUs some shapes need more, and fits_scratch rejects them (the
// entry point then returns SQ_ERR_UNSUPPORTED without launching).
static void check_static_scratch() {
    const long long cap = 40ll * 1024 * 1024;
    const long long Ms[] = {1, 128, 256, 512, 1000, 2048, 4096};
    const long long Ns[] = {1, 256, 512, 1024, 4096};
    const long long Ks[] = {2048, 4096, 8192};
    for (int sms : {2, 148, 152, 159, 160, 200, 256}) {
        long long worst = 0;
        for (long long M : Ms)
            for (long long N : Ns)
                for (long long K : Ks) {
                    int grid = 0;
                    const long long need = sk_workspace_bytes(plan_launch(M, N, K, sms, true, &grid));
                    if (need > worst) worst = need;
                    CHECK(fits_scratch(need, cap) == (need <= cap), "fits_scratch(%lld)", need);
                }
        // the largest split uses every SM: sms / 4 tiles of 128 x 256, four pieces each
        if (sms % 4 == 0) {
            int grid = 0;
            const Schedule sc = plan_launch(128ll * (sms / 4), 256, 4096, sms, true, &grid);
            CHECK(sc.sk_ctas == sms, "sms %d: %d split CTAs", sms, sc.sk_ctas);
            const long long need = sk_workspace_bytes(sc);
            if (need > worst) worst = need;
        }
        if (sms <= 159) CHECK(fits_scratch(worst, cap), "sms %d: worst split %lld > %lld", sms, worst, cap);
        if (sms >= 160) CHECK(!fits_scratch(worst, cap), "sms %d: every split fits (%lld)", sms, worst);
        // the counter block is one size per device, at the workspace's start
        CHECK(sk_counter_bytes_on(sms) % 256 == 0 && sk_counter_bytes_on(sms) >= sms * 64ll,
              "counter block on %d SMs", sms);
        ++g_checked;
    }
}

int main() {
    check_static_scratch();
    const long long Ms[] = {1, 127, 128, 129, 255, 256, 300, 1000, 2560, 8192};
    const long long Ns[] = {1, 255, 256, 257, 1000, 1024, 2304, 3072, 4096};
    const long long Ks[] = {16, 1024, 1040, 2048, 2080, 4096, 8192};
    const int sms[] = {1, 2, 7, 148, 152};
    for (long long M : Ms)
        for (long long N : Ns)
            for (int s : sms) {
                for (long long K : Ks)
                    for (int split = 0; split < 2; ++split) check_one_cta(M, N, K, s, split != 0);
                check_pair(M, N, s / 2 > 0 ? s / 2 : 1);
                check_pair(M, N, 76);
            }
    std::printf("checked %lld launches, %lld failures\n", g_checked, g_fail);
    return g_fail ? 1 : 0;
}
