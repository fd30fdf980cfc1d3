// planner_check.cu -- host-only check of the decode matvec planner (plan_gemv):
// for every format, a sweep of widths, row counts, vector counts, both
// activation kinds and both callers (the matvec and the expert matvec), each
// accepted plan must satisfy what the kernels assume.
// Built and run by tests/test_planner_host.py; no GPU is touched.
#include <cstdio>

#include "gemv_launch.cuh"

using namespace qmv;

template <int T>
static int check(const char* name, const int64_t* cols_list, int n_cols, int* accepted)
{
    using F = Fmt<T>;
    const int64_t rows_list[] = {1, 7, 37, 128, 896, 1152, 4096, 9728, 151936, 1 << 20};
    const int nvs[] = {1, 2, 3, 4, 5, 8, 9, 16, 17, 64};
    int bad = 0;
    auto fail = [&](const char* what, int64_t rows, int64_t cols, int nv, bool a8) {
        std::printf("%s rows=%lld cols=%lld n_vec=%d a8=%d: %s\n", name, (long long)rows, (long long)cols, nv, (int)a8,
                    what);
        ++bad;
    };
    for (int ci = 0; ci < n_cols; ++ci)
        for (int64_t rows : rows_list)
            for (int nv : nvs)
                for (int a = 0; a < 4; ++a) {
                    const int64_t cols = cols_list[ci];
                    const bool a8 = (a & 1) != 0;
                    // a < 2: as the matvec plans (up to 4 rows per warp, at least one tile per SM);
                    // a >= 2: as the expert matvec plans (rows per warp capped at the decode width)
                    const int g16 = nv < 16 ? nv : 16;
                    GemvPlan pl{};
                    const bool ok = a < 2 ? plan_gemv<T>(a8, rows, cols, nv, pl, 4, 152)
                                          : plan_gemv<T>(a8, rows, cols, g16, pl, rows_in_flight_rt(T, g16, false));
                    if (!ok) continue;   // refused: shared memory
                    ++*accepted;
                    const int nb = (int)(cols / F::BS);
                    const size_t tr = (size_t)kConsumerWarps * pl.rpw;
                    const size_t base = 256 + (((size_t)pl.xhat_bytes + 127) & ~size_t(127));
                    if (pl.smem != base + (size_t)pl.stages * pl.seg_cap * tr) fail("smem is not base + S stages", rows, cols, nv, a8);
                    if (pl.smem > kSmemOnePerSm) fail("more shared memory than a CTA may have", rows, cols, nv, a8);
                    if (pl.stages < 2 || pl.stages > kMaxStages) fail("stage count outside 2..8", rows, cols, nv, a8);
                    if (pl.kb < 1 || (int64_t)pl.n_chunks * pl.kb < nb || (int64_t)(pl.n_chunks - 1) * pl.kb >= nb)
                        fail("chunks do not cover the row exactly", rows, cols, nv, a8);
                    if (pl.seg_cap % 16 || pl.seg_cap < (uint32_t)(pl.kb * F::BB + 30))
                        fail("row segment cannot hold a chunk's 16-byte-aligned superset", rows, cols, nv, a8);
                    if (pl.group < 1 || pl.group > 16 || pl.group > nv) fail("vector group outside 1..16", rows, cols, nv, a8);
                    if (pl.xhat_bytes != xhat_bytes(T, a8, pl.group, (int)cols)) fail("staged activations mis-sized", rows, cols, nv, a8);
                    if (pl.group > 1 && pl.xhat_bytes > kXhatMaxBytes) fail("staged activations over the limit", rows, cols, nv, a8);
                    if (pl.rpw != 1 && pl.rpw != 2 && pl.rpw != 4) fail("rows per warp not 1, 2 or 4", rows, cols, nv, a8);
                    if (pl.n_chunks > 1 && pl.rpw > rows_in_flight_rt(T, pl.group, true))
                        fail("a multi-chunk row group wider than the decode width", rows, cols, nv, a8);
                }
    return bad;
}

// The plain bf16 GEMM's tile width model against the faster width of A/B runs
// of both widths on a 152-SM GB300 (BF16 rows), and two limits: a single
// 128-token tile for at most 128 tokens, 256-token tiles when they fill whole
// waves without padding.
static int check_gemm_bf16_width()
{
    struct Case { int64_t rows, m; bool narrow; };
    const Case cases[] = {{14336, 512, true},  {14336, 768, false}, {14336, 1024, false}, {14336, 1536, false},
                          {14336, 2048, false}, {4096, 512, true},   {4096, 1024, false}};
    int bad = 0;
    for (const Case& c : cases)
        if (gemm_bf16_narrow(c.rows, c.m, 152) != c.narrow) {
            std::printf("bf16 GEMM width: rows=%lld m=%lld picks %d tokens\n", (long long)c.rows, (long long)c.m,
                        gemm_bf16_narrow(c.rows, c.m, 152) ? 128 : 256);
            ++bad;
        }
    for (int64_t rows : {128, 4096, 14336, 151936})
        for (int64_t m : {1, 64, 127, 128})
            if (!gemm_bf16_narrow(rows, m, 152)) { std::printf("bf16 GEMM width: m=%lld not 128\n", (long long)m); ++bad; }
    if (gemm_bf16_narrow(152 * 128, 256 * 3, 152)) { std::printf("bf16 GEMM width: whole waves not 256\n"); ++bad; }
    return bad;
}

int main()
{
    const int64_t c32[] = {32, 96, 896, 2880, 4096, 4864, 8288, 14336, 32768, 65536};
    const int64_t c256[] = {256, 512, 4096, 14336, 32768, 65536};
    int accepted = 0, bad = 0;
    bad += check<QMV_Q4_0>("Q4_0", c32, 10, &accepted);
    bad += check<QMV_Q5_0>("Q5_0", c32, 10, &accepted);
    bad += check<QMV_Q8_0>("Q8_0", c32, 10, &accepted);
    bad += check<QMV_MXFP4>("MXFP4", c32, 10, &accepted);
    bad += check<QMV_Q4_K>("Q4_K", c256, 6, &accepted);
    bad += check<QMV_Q6_K>("Q6_K", c256, 6, &accepted);
    bad += check_gemm_bf16_width();
    std::printf("plans accepted %d, violations %d\n", accepted, bad);
    return bad ? 1 : 0;
}
