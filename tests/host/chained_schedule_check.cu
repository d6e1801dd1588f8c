// Host-side check of the chained k-split schedule (SkPlan, sk_schedule in
// gemm_kernels.cuh), compiled by tests/test_chained_schedule_host.py.  For
// many (tiles, k-slices, workers) it walks every worker's segments exactly as
// the kernel does and checks that
//   - every (tile, slice) is run exactly once;
//   - a worker has at most one head (a tile begun at slice 0 and not finished)
//     and one tail (a tile continued to its last slice), and worker w's tail
//     continues exactly the tile and slice where worker w-1's head stopped;
//   - no worker's tail comes before, in its own slice count, the point where
//     worker w-1 has finished that head (so no worker ever waits on a head
//     that is still being computed when all run at one speed);
//   - the heads' scratch and flag indices stay below `workers`.
// Prints "ok <cases>" or the first violation, and exits non-zero on one.
#include <cstdio>
#include <vector>

#include "gemm_kernels.cuh"

using repops::gemm::SkArgs;
using repops::gemm::SkPlan;
using repops::gemm::SkSeg;

static int check(int64_t tiles, int kt, int workers) {
    SkArgs sk{};
    repops::gemm::sk_schedule(tiles, kt, workers, sk);
    std::vector<int> cover(size_t(tiles) * kt, -1);
    std::vector<int64_t> head_tile(workers, -1), head_end(workers, -1), head_done(workers, -1);
    for (int w = 0; w < workers; ++w) {
        const SkPlan plan(sk, w, workers);
        int64_t slices = 0;
        int heads = 0, tails = 0;
        for (int s = 0; s < plan.nseg; ++s) {
            const SkSeg g = plan.seg(s);
            if (g.tile < 0 || g.tile >= tiles || g.kb < 0 || g.kb >= g.ke || g.ke > kt) {
                std::printf("bad segment tiles=%lld kt=%d workers=%d w=%d\n", (long long)tiles, kt, workers, w);
                return 1;
            }
            if ((g.kind == 1 && (g.kb != 0 || g.ke != kt)) || (g.kind == 0 && (g.kb != 0 || g.ke == kt)) ||
                (g.kind == 2 && (g.kb == 0 || g.ke != kt || w == 0))) {
                std::printf("bad kind tiles=%lld kt=%d workers=%d w=%d\n", (long long)tiles, kt, workers, w);
                return 1;
            }
            for (int k = g.kb; k < g.ke; ++k) {
                int &c = cover[size_t(g.tile) * kt + k];
                if (c != -1) {
                    std::printf("slice run twice tiles=%lld kt=%d workers=%d\n", (long long)tiles, kt, workers);
                    return 1;
                }
                c = w;
            }
            slices += g.ke - g.kb;
            if (g.kind == 0) {
                ++heads;
                head_tile[w] = g.tile;
                head_end[w] = g.ke;
                head_done[w] = slices;
            }
            if (g.kind == 2) ++tails;
        }
        if (heads > 1 || tails > 1) {
            std::printf("several heads or tails tiles=%lld kt=%d workers=%d w=%d\n", (long long)tiles, kt, workers, w);
            return 1;
        }
    }
    for (int64_t i = 0; i < tiles * kt; ++i)
        if (cover[size_t(i)] < 0) {
            std::printf("slice never run tiles=%lld kt=%d workers=%d\n", (long long)tiles, kt, workers);
            return 1;
        }
    for (int w = 1; w < workers; ++w) {
        const SkPlan plan(sk, w, workers);
        int64_t before = 0;
        for (int s = 0; s < plan.nseg; ++s) {
            const SkSeg g = plan.seg(s);
            if (g.kind == 2) {
                if (head_tile[w - 1] != g.tile || head_end[w - 1] != g.kb) {
                    std::printf("tail does not continue the previous head tiles=%lld kt=%d workers=%d w=%d\n",
                                (long long)tiles, kt, workers, w);
                    return 1;
                }
                if (before < head_done[w - 1]) {
                    std::printf("tail before the head is done tiles=%lld kt=%d workers=%d w=%d\n",
                                (long long)tiles, kt, workers, w);
                    return 1;
                }
            }
            before += g.ke - g.kb;
        }
    }
    return 0;
}

int main() {
    long cases = 0;
    const int kts[] = {1, 2, 3, 7, 32, 64, 94, 256};
    for (int64_t tiles = 1; tiles <= 80; ++tiles)
        for (int workers = 1; workers <= tiles; ++workers)
            for (int kt : kts) {
                if (check(tiles, kt, workers)) return 1;
                ++cases;
            }
    const int64_t big[] = {256, 512, 1024, 1536, 2048, 8192};
    const int ws[] = {1, 7, 100, 151, 152, 255, 303, 304};
    for (int64_t tiles : big)
        for (int workers : ws)
            for (int kt : kts) {
                if (workers > tiles) continue;
                if (check(tiles, kt, workers)) return 1;
                ++cases;
            }
    std::printf("ok %ld\n", cases);
    return 0;
}
