// Work schedules of the tcgen05 GEMM kernels: which output tiles (and which
// K-block ranges of them) each persistent CTA or CTA pair processes, and the
// split-K workspace layout.  Plain functions of the launch shape -- the CTA
// index and grid size are arguments -- so that the host can plan launches and
// check the schedules' invariants without a GPU.
#pragma once
#include <cstdint>

namespace sq {
namespace sched {

constexpr int BM = 128, BN = 256, BK = 64;  // output tile rows, columns; K block (bf16 elements)
constexpr int KB_PER_CHUNK = 16;            // 16 * 64 = 1024 K per exact fp32 chunk
constexpr int NUM_EPI_WARPS = 8;

// Work units of a launch.  Two schedules:
//
// Whole tiles (no workspace).  The BM x BN tiles that fill whole waves of the
// persistent grid are units as they are; when the last, partial wave holds at
// most half a wave of tiles, each of them is cut into two 128-column halves
// (MMA N = 128), so that the last round takes half as long.  (Quarters, N = 64,
// measured slower: the A tile is loaded in full for a quarter of the work.)
//
// Split K (a workspace is given).  The K blocks of the last sk_tiles tiles
// form one range, cut evenly over sk_ctas CTAs (a CTA's share may cover the
// end of one tile and the start of the next).  A piece of a tile (a K-block
// range of it) leaves its exact int32 partial sums in the workspace; the CTA
// whose piece of the tile completes last adds the others' partials to its own
// and runs the epilogue.  Measured on GB300, the partials' round trip through
// L2 (about 4 us on the finishing CTA's path) costs more than a split saves
// unless the tiles are fewer than the SMs and long in K, so the split is used
// only there: every tile cut into `pieces` <= 4 equal K ranges of at least
// 1024, one per CTA (small M with a large K: a few tiles would otherwise keep
// a few SMs busy for the whole K).
//
// Tiles are numbered m-fastest, so CTAs working at the same time share B tiles
// in L2.
constexpr int kMinSplitKb = 32;  // split K only for K >= 2048 (32 blocks of 64)
constexpr int kMaxPieces = 4;

struct Schedule {
    int m_tiles, nkb;
    int full_items, sub, items;      // whole-tile schedule (halves in the last wave)
    int dp_tiles, sk_tiles, sk_ctas;  // split-K part; sk_tiles == 0: not used
    int sk_cnt_tiles;                 // tiles the counter block has room for (2 x grid)
};

__host__ __device__ inline Schedule make_schedule(int m_tiles, int n_tiles, int nkb, int grid,
                                                  bool split_k) {
    Schedule sc;
    sc.m_tiles = m_tiles;
    sc.nkb = nkb;
    const int tiles = m_tiles * n_tiles;
    const int waves = tiles / grid, rem = tiles - waves * grid;
    sc.sub = (waves >= 1 && rem > 0 && 2 * rem <= grid) ? 2 : 1;
    sc.full_items = sc.sub == 1 ? tiles : waves * grid;
    sc.items = sc.full_items + (tiles - sc.full_items) * sc.sub;
    sc.dp_tiles = tiles;
    sc.sk_tiles = 0;
    sc.sk_ctas = 0;
    sc.sk_cnt_tiles = 0;
    if (split_k && waves == 0 && nkb >= kMinSplitKb) {
        // fewer tiles than SMs and a long K: cut every tile into `pieces`
        // equal K ranges, one per CTA
        int pieces = grid / tiles;
        if (pieces > kMaxPieces) pieces = kMaxPieces;
        if (pieces >= 2) {
            sc.sub = 1;
            sc.sk_tiles = tiles;
            sc.dp_tiles = 0;
            sc.sk_ctas = tiles * pieces;
            sc.sk_cnt_tiles = grid;  // >= tiles
            sc.full_items = sc.items = 0;
        }
    }
    return sc;
}

// First K-block index (over the split tiles' concatenated K blocks) of CTA c's share.
__host__ __device__ inline long long sk_start(const Schedule &sc, int c) {
    return (long long)c * ((long long)sc.sk_tiles * sc.nkb) / sc.sk_ctas;
}

// The CTA whose share holds K-block index `it`: the largest c with sk_start(c) <= it.
__host__ __device__ inline int sk_cta_of(const Schedule &sc, long long it) {
    const long long total = (long long)sc.sk_tiles * sc.nkb;
    long long c = (it * sc.sk_ctas + sc.sk_ctas - 1) / total;
    if (c > sc.sk_ctas - 1) c = sc.sk_ctas - 1;
    if (sk_start(sc, (int)c) > it) --c;
    return (int)c;
}

struct Work {
    int m0, n0, bn;
    int kb0, kb1;  // K blocks [kb0, kb1) of the tile
    int skt;       // split tile index of a piece, -1 for a whole tile
};

// Walks one CTA's units: its whole-tile items, then the pieces of its share
// (K-block indices fit in 32 bits: at most 2 x grid tiles of 2081 blocks).
struct Cursor {
    int i, it, end;
};

// CTA `cta`'s cursor (in a kernel: blockIdx.x).
__host__ __device__ __forceinline__ void cursor_init(const Schedule &sc, Cursor &cu, int cta) {
    cu.i = cta;
    cu.it = cu.end = 0;
    if (sc.sk_tiles > 0 && cta < sc.sk_ctas) {
        cu.it = (int)sk_start(sc, cta);
        cu.end = (int)sk_start(sc, cta + 1);
    }
}

// The next unit of a CTA of a `grid`-CTA launch (in a kernel: gridDim.x).
__host__ __device__ __forceinline__ bool next_work(const Schedule &sc, Cursor &cu, Work &w,
                                                   int grid) {
    if (cu.i < sc.items) {
        const int i = cu.i;
        cu.i += grid;
        w.kb0 = 0;
        w.kb1 = sc.nkb;
        w.skt = -1;
        if (i < sc.full_items) {
            w.m0 = (i % sc.m_tiles) * BM;
            w.n0 = (i / sc.m_tiles) * BN;
            w.bn = BN;
        } else {
            const int j = i - sc.full_items;
            const int t = sc.full_items + j / sc.sub;
            w.bn = BN / sc.sub;
            w.m0 = (t % sc.m_tiles) * BM;
            w.n0 = (t / sc.m_tiles) * BN + (j % sc.sub) * w.bn;
        }
        return true;
    }
    if (cu.it >= cu.end) return false;
    const int r = cu.it / sc.nkb;
    const int tb = r * sc.nkb;
    w.kb0 = cu.it - tb;
    w.kb1 = min(sc.nkb, cu.end - tb);
    const int t = sc.dp_tiles + r;
    w.m0 = (t % sc.m_tiles) * BM;
    w.n0 = (t / sc.m_tiles) * BN;
    w.bn = BN;
    // -1: the whole tile lies in this share
    w.skt = (w.kb0 == 0 && w.kb1 == sc.nkb) ? -1 : r;
    cu.it = tb + sc.nkb;
    return true;
}

// Workspace of the split-K schedule: two counters per (tile, epilogue warp) --
// pieces that finished their MMAs, pieces whose partials are written -- then,
// per CTA, two partial slots (the first and the last piece of its share), each
// NUM_EPI_WARPS sub-blocks of 32 rows x 128 columns of int32.  The counter
// block has one size for every shape on a device (room for 2 x grid tiles), so
// that the counters of one launch never fall on another launch's partial slots
// in a shared workspace.
constexpr int kSlotWarpBytes = 32 * 128 * 4;
__host__ __device__ inline long long sk_counter_bytes(const Schedule &sc) {
    return ((long long)sc.sk_cnt_tiles * NUM_EPI_WARPS * 2 * 4 + 255) / 256 * 256;
}
__host__ __device__ inline long long sk_workspace_bytes(const Schedule &sc) {
    if (sc.sk_tiles == 0) return 0;
    return sk_counter_bytes(sc) + (long long)sc.sk_ctas * 2 * NUM_EPI_WARPS * kSlotWarpBytes;
}
// The counter block on a GPU of `sms` SMs (one size for every split shape there).
__host__ __device__ inline long long sk_counter_bytes_on(int sms) {
    Schedule sc{};
    sc.sk_cnt_tiles = sms;
    return sk_counter_bytes(sc);
}
// Whether a launch that needs `need` workspace bytes runs on a fixed scratch
// of `capacity` bytes (the static scratch of sq_linear_i8_static_ws).
inline bool fits_scratch(long long need, long long capacity) { return need <= capacity; }

// Work items of the pair kernel: 256 x 256 pair tiles, numbered n-fastest, so
// that the clusters of a wave work on all column tiles of a few row blocks and
// every row block of A is read from DRAM once (the weights, a few MB, stay in
// L2); when the last, partial wave holds at most half the clusters, each of its
// tiles is cut into two 256 x 128 halves (MMA N = 128, 64 rows of B per CTA):
// one round of halves then replaces the round of whole tiles.  (With more
// than half the clusters busy, halves would need two rounds, and a half
// tile, which reads as much of A as a whole one for half the products, takes
// well over half a tile's time: measured slower on GB300.)  A launch with at
// most half as many tiles as clusters runs all its tiles as halves, on twice
// the clusters.
struct PairSchedule {
    int m_pairs, n_tiles, full_items, sub, items;
};

__host__ __device__ inline PairSchedule make_pair_schedule(int m_pairs, int n_tiles,
                                                           int clusters) {
    PairSchedule sc;
    sc.m_pairs = m_pairs;
    sc.n_tiles = n_tiles;
    const int tiles = m_pairs * n_tiles;
    const int waves = tiles / clusters, rem = tiles - waves * clusters;
    sc.sub = (rem > 0 && 2 * rem <= clusters) ? 2 : 1;  // waves = 0: 2 tiles <= clusters
    sc.full_items = sc.sub == 1 ? tiles : waves * clusters;
    sc.items = sc.full_items + (tiles - sc.full_items) * sc.sub;
    return sc;
}

// item i: pair rows from m0 (256), columns n0.. of width bn (256 or 128)
__host__ __device__ __forceinline__ void pair_item_at(const PairSchedule &sc, int i, int &m0, int &n0,
                                             int &bn) {
    if (i < sc.full_items) {
        n0 = (i % sc.n_tiles) * BN;
        m0 = (i / sc.n_tiles) * 2 * BM;
        bn = BN;
    } else {
        const int j = i - sc.full_items;
        const int t = sc.full_items + j / sc.sub;
        bn = BN / sc.sub;
        n0 = (t % sc.n_tiles) * BN + (j % sc.sub) * bn;
        m0 = (t / sc.n_tiles) * 2 * BM;
    }
}


// Schedule of an M x N x K launch on `sms` SMs, and the grid it runs on.
inline Schedule plan_launch(int64_t M, int64_t N, int64_t K, int sms, bool split_k, int *grid) {
    const int m_tiles = (int)((M + BM - 1) / BM), n_tiles = (int)((N + BN - 1) / BN);
    const int nkb = (int)((K + BK - 1) / BK);
    const int tiles = m_tiles * n_tiles;
    if (split_k) {
        const Schedule sc = make_schedule(m_tiles, n_tiles, nkb, sms, true);
        if (sc.sk_tiles > 0) {
            *grid = sc.dp_tiles > 0 ? sms : sc.sk_ctas;
            return sc;
        }
    }
    *grid = tiles < sms ? tiles : sms;
    return make_schedule(m_tiles, n_tiles, nkb, *grid, false);
}

}  // namespace sched
}  // namespace sq
