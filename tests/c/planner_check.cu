// Host-side checks of the kernel-mapping rules (make_plan and its helpers)
// on a stand-in device description: 152 SMs and segment-kernel occupancies
// of 2048 / threads / 2 CTAs per SM.  Only host code runs; no device needed.
// Each expectation restates a rule that the library's comments give with
// the measurement behind it.
#include <cstdio>

#include "../../log_sum_exp_gb300/csrc/lse_api.cu"

namespace {

int g_fail = 0;

void expect(bool ok, const char* what) {
    if (!ok) {
        std::printf("FAIL: %s\n", what);
        ++g_fail;
    }
}

lse::DeviceInfo fake_device() {
    lse::DeviceInfo info;
    info.ready = true;
    info.sms = 152;
    for (int dt = 0; dt < 3; ++dt)
        for (int v = 0; v < 2; ++v)
            for (int t = 0; t < 5; ++t) info.seg_occ[dt][v][t] = 2048 / (32 << t) / 2;
    return info;
}

const void* const kAligned = reinterpret_cast<const void*>(static_cast<uintptr_t>(1) << 20);

lse_plan plan(lse_dtype dt, int64_t B, int64_t N, int64_t rs, const void* x = kAligned,
              const lse_plan* req = nullptr, bool logprob = false, bool e16 = false,
              lse_status* st = nullptr) {
    static const lse::DeviceInfo info = fake_device();
    lse_plan p;
    std::memset(&p, 0, sizeof p);
    const lse_status s = lse::make_plan(x, dt, B, N, rs, info, req, logprob, &p, e16);
    if (st) *st = s;
    else expect(s == LSE_OK, "make_plan returned an error");
    return p;
}

}  // namespace

int main() {
    // Back-to-back rows of 16..128 bytes: the vector ring where it measured
    // faster (every width but f32 rows of 2 vectors), else the sub-warp kernel.
    lse_plan p = plan(LSE_F32, 1 << 20, 32, 32);
    expect(p.path == LSE_PATH_ROWTILE && p.slots_per_lane == 8 && p.threads == 768 && p.grid == 152,
           "f32 rows of 128 bytes: ring, 8 vectors, one CTA of 24 warps per SM");
    p = plan(LSE_BF16, 1 << 20, 64, 64);
    expect(p.path == LSE_PATH_ROWTILE && p.slots_per_lane == 8, "bf16 rows of 128 bytes: ring, 8 vectors");
    p = plan(LSE_F32, 1 << 22, 8, 8);
    expect(p.path == LSE_PATH_SUBWARP && p.lanes_per_row == 1 && p.slots_per_lane == 2,
           "f32 rows of 32 bytes: sub-warp, 1 lane x 2 vectors");
    p = plan(LSE_F32, 1 << 20, 32, 36);
    expect(p.path == LSE_PATH_SUBWARP, "rows not back to back: no ring");
    p = plan(LSE_F32, 1000, 32, 32);
    expect(p.path == LSE_PATH_SUBWARP, "too few rows for every CTA: no ring");

    // Other widths of 32..128 bytes: the any-width ring, a thread per row (row
    // value and token log-probability, not the 16-bit exponentials); shorter
    // rows stay on the sub-warp kernel.
    p = plan(LSE_F32, 1 << 22, 13, 13);
    expect(p.path == LSE_PATH_ROWTILE && p.slots_per_lane == 0 && p.lanes_per_row == 1 &&
               p.vector_bytes == 1,
           "f32 rows of 52 bytes: any-width ring, a thread per row");
    p = plan(LSE_F32, 1 << 22, 13, 13, kAligned, nullptr, true);
    expect(p.path == LSE_PATH_ROWTILE && p.lanes_per_row == 1, "token log-probability: the same ring");
    p = plan(LSE_F32, 1 << 22, 13, 13, kAligned, nullptr, false, true);
    expect(p.path == LSE_PATH_SUBWARP, "16-bit exponentials: sub-warp kernel");
    p = plan(LSE_F32, 1 << 22, 13, 14);
    expect(p.path == LSE_PATH_SUBWARP, "strided rows: sub-warp kernel");
    p = plan(LSE_F32, 1 << 22, 7, 7);
    expect(p.path == LSE_PATH_SUBWARP, "f32 rows of 28 bytes: sub-warp kernel");

    // Longer back-to-back rows: the grouped ring where a quarter or more of the
    // sub-warp slots would be empty (rows just past a power of two of slots),
    // for f32 rows and 16-bit rows of at most 1.5 KB, or where the sub-warp
    // kernel cannot hold the row.
    p = plan(LSE_F32, 1 << 20, 129, 129);
    expect(p.path == LSE_PATH_ROWTILE && p.lanes_per_row == 4, "f32 N=129: grouped ring, 4 lanes");
    // One thread per row up to 128 bytes plus one element: f32 N = 33
    // (132 bytes, at most 9 vectors from any 4-byte offset), bf16 N = 65.
    p = plan(LSE_F32, 1 << 20, 33, 33);
    expect(p.path == LSE_PATH_ROWTILE && p.lanes_per_row == 1 && p.vector_bytes == 1,
           "f32 N=33: the ring, a thread per row");
    p = plan(LSE_BF16, 1 << 20, 65, 65);
    expect(p.path == LSE_PATH_ROWTILE && p.lanes_per_row == 1, "bf16 N=65: the ring, a thread per row");
    p = plan(LSE_BF16, 1 << 20, 66, 66);
    expect(!(p.path == LSE_PATH_ROWTILE && p.lanes_per_row == 1), "bf16 N=66: not a thread per row");
    p = plan(LSE_F32, 1 << 20, 520, 520);
    expect(p.path == LSE_PATH_ROWTILE && p.lanes_per_row == 16, "f32 N=520: grouped ring, 16 lanes");
    p = plan(LSE_F32, 1 << 20, 300, 300);
    expect(p.path == LSE_PATH_SUBWARP, "f32 N=300 (80 % of the slots full): sub-warp kernel");
    p = plan(LSE_BF16, 1 << 20, 1025, 1025);
    expect(p.path == LSE_PATH_SUBWARP, "bf16 N=1025 (2 KB rows): sub-warp kernel");
    p = plan(LSE_BF16, 1 << 18, 2047, 2047);
    expect(p.path == LSE_PATH_ROWTILE && p.lanes_per_row == 16, "bf16 N=2047: grouped ring, 16 lanes");
    p = plan(LSE_F32, 1 << 20, 68, 68);
    expect(p.path == LSE_PATH_SUBWARP, "rows of <= 512 bytes: no grouped ring");
    p = plan(LSE_F32, 1 << 20, 129, 129, kAligned, nullptr, false, true);
    expect(p.path == LSE_PATH_SUBWARP && p.lanes_per_row == 8 && p.slots_per_lane == 6,
           "f32 N=129 with 16-bit exponentials: 8 lanes x 6 slots (32 vectors + 2 edge slots)");

    // Sub-warp shapes: fewest lanes with <= 4 slots; vector rows of more than
    // 16 slots take half the lanes with up to 8 slots each; slots per lane are
    // 1, 2, 3, 4, 6 or 8 (5 and 7 too for a whole warp).
    p = plan(LSE_F32, 1 << 20, 40, 44);
    expect(p.path == LSE_PATH_SUBWARP && p.lanes_per_row == 4 && p.slots_per_lane == 3,
           "f32 N=40: 4 lanes x 3 slots");
    p = plan(LSE_F32, 1 << 20, 128, 128);
    expect(p.path == LSE_PATH_SUBWARP && p.lanes_per_row == 4 && p.slots_per_lane == 8,
           "f32 N=128: 4 lanes x 8 slots");
    p = plan(LSE_F32, 1 << 17, 1001, 1001);
    expect(p.path == LSE_PATH_SUBWARP && p.lanes_per_row == 32 && p.slots_per_lane == 8,
           "f32 N=1001 (250 vectors + 2 peel slots): a warp x 8 slots");
    // A whole warp per row takes 5 and 7 slots per lane too (row stride 1040
    // elements keeps the rows strided, off the bulk-copy rings).
    p = plan(LSE_BF16, 1 << 16, 1025, 1040);
    expect(p.path == LSE_PATH_SUBWARP && p.lanes_per_row == 32 && p.slots_per_lane == 5,
           "bf16 N=1025 (128 vectors + 2 slots): a warp x 5 slots");
    p = plan(LSE_BF16, 1 << 16, 1700, 1704);
    expect(p.path == LSE_PATH_SUBWARP && p.lanes_per_row == 32 && p.slots_per_lane == 7,
           "bf16 N=1700 (212 vectors + 2 slots): a warp x 7 slots");
    p = plan(LSE_F32, 1 << 16, 520, 520);
    expect(p.path == LSE_PATH_ROWTILE && p.lanes_per_row == 16,
           "f32 N=520 back to back (132 slots): the grouped ring, as measured against 6 slots");
    expect(lse::subwarp_auto_slots(33, true) == 48 && lse::subwarp_auto_slots(32, true) == 32 &&
               lse::subwarp_auto_slots(18, true) == 24 && lse::subwarp_auto_slots(10, true) == 12,
           "sub-warp slot counts");

    // Long rows: a CTA per row, split when the rows cannot fill the GPU.
    p = plan(LSE_F32, 512, 128256, 128256);
    expect(p.path == LSE_PATH_CTA && p.threads == 512 && p.splits == 1, "512 x 128256 f32: CTA 512");
    p = plan(LSE_BF16, 8192, 32000, 32000);
    expect(p.path == LSE_PATH_CTA && p.threads == 128 && p.splits == 1, "8192 x 32000 bf16: CTA 128");
    p = plan(LSE_F32, 16, 16777216, 16777216);
    expect(p.path == LSE_PATH_SPLIT && p.threads == 512 && p.splits == 128 && p.launches == 2 &&
               p.scratch_bytes == 16 * 128 * 8,
           "16 x 16.7M f32: 128 splits of 512 threads and a merge");

    // Fewer rows than SMs: 128 threads where one full batch each covers the
    // row, else at least 256.
    p = plan(LSE_F32, 64, 4096, 4096);
    expect(p.path == LSE_PATH_CTA && p.threads == 128 && p.splits == 1 && p.grid == 64,
           "64 x 4096 f32: a CTA of 128 per row, one batch per thread");
    p = plan(LSE_F32, 64, 8192, 8192);
    expect(p.path == LSE_PATH_CTA && p.threads == 256, "64 x 8192 f32: a CTA of 256 per row");

    // Alignment: rows off a 16-byte boundary keep vectors (peeled); a base
    // that is not element aligned gets element loads.
    p = plan(LSE_F32, 64, 4096, 4096, reinterpret_cast<const void*>((1u << 20) + 4));
    expect(p.vector_bytes == 16, "f32 rows 4 bytes off a boundary: vectors with a peel");
    p = plan(LSE_F32, 64, 4096, 4096, reinterpret_cast<const void*>((1u << 20) + 2));
    expect(p.vector_bytes == 1, "a base that is not element aligned: element loads");

    // Requests.
    lse_status st;
    lse_plan req;
    std::memset(&req, 0, sizeof req);
    req.path = LSE_PATH_ROWTILE;
    plan(LSE_F32, 1 << 20, 5, 6, kAligned, &req, false, false, &st);
    expect(st == LSE_ERR_INVALID_ARG, "forced ring on strided rows: invalid");
    req.path = LSE_PATH_SUBWARP;
    req.lanes_per_row = 2;
    plan(LSE_F32, 1 << 20, 80, 80, kAligned, &req, false, false, &st);
    expect(st == LSE_ERR_INVALID_ARG, "2 lanes for 20 slots (10 each): invalid");
    req.lanes_per_row = 4;
    p = plan(LSE_F32, 1 << 20, 80, 80, kAligned, &req, false, false, &st);
    expect(st == LSE_OK && p.slots_per_lane == 6, "4 lanes for 20 slots: 6 slots each");
    req.path = LSE_PATH_SPLIT;
    req.lanes_per_row = 0;
    req.splits = 3;
    p = plan(LSE_F32, 4, 4096, 4096, kAligned, &req, false, false, &st);
    expect(st == LSE_OK && p.path == LSE_PATH_SPLIT && p.splits == 3, "forced 3 splits");
    p = plan(LSE_F32, 7, 0, 0);
    expect(p.path == LSE_PATH_EMPTY && p.launches == 1, "N = 0: the fill kernel");

    // Row backward: vectors, peeled vectors, the flat array or elements;
    // flattened short rows; threads across a row = ceil(slots / 4).
    {
        const lse::DeviceInfo info = fake_device();
        const char* base = static_cast<const char*>(kAligned);
        auto bwd = [&](int eb, int64_t B, int64_t N, int64_t rs, const void* x, const void* dx,
                       int64_t drs, lse::BackwardArgs* a) {
            int mode = -1;
            expect(lse::plan_backward(x, eb, B, N, rs, dx, drs, info, a, &mode) == LSE_OK,
                   "plan_backward returned an error");
            return mode;
        };
        lse::BackwardArgs a;
        const void* dx = base + (64 << 20);
        int m = bwd(4, 1 << 20, 32, 32, base, dx, 32, &a);
        expect(m == lse::kBwdVector && a.small && a.block.x == 256,
               "f32 rows of 8 vectors: flattened short rows");
        m = bwd(4, 512, 128256, 128256, base, dx, 128256, &a);
        expect(m == lse::kBwdVector && !a.small && a.block.x == 256 && a.block.y == 1 &&
                   a.seg_slots == 4096 && a.grid.x == 8 && a.grid.y == 512,
               "512 x 128256 f32: 256 threads per row, 8 segments of 4096 vectors");
        m = bwd(4, 1 << 20, 129, 129, base, dx, 129, &a);
        expect(m == lse::kBwdFlat && a.grid.x == 152 * 4 && a.block.x == 256,
               "f32 N=129 back to back: the flat array, one wave");
        m = bwd(4, 1335, 50257, 50257, base, dx, 50257, &a);
        expect(m == lse::kBwdPeel && a.block.x == 256, "f32 N=50257 (rows over 16 KB): peeled rows");
        m = bwd(4, 1335, 1001, 1001, base, base + (64 << 20) + 4, 1001, &a);
        expect(m == lse::kBwdScalar, "dx at another offset from a boundary than x: elements");
        m = bwd(4, 4096, 13, 14, base, dx, 14, &a);
        expect(m == lse::kBwdScalar, "f32 N=13 (3 vectors), not back to back: elements");
        m = bwd(2, 4096, 9, 9, base, dx, 9, &a);
        expect(m == lse::kBwdFlat, "bf16 N=9 back to back: the flat array");
        m = bwd(2, 4096, 5, 5, base, dx, 5, &a);
        expect(m == lse::kBwdScalar && !a.small && a.block.x == 2 && a.block.y == 128,
               "bf16 N=5: elements, 2 threads across a row");
        m = bwd(4, 1 << 16, 132, 133, base, dx, 133, &a);
        expect(m == lse::kBwdPeel && a.block.x == 9 && a.block.y == 28,
               "f32 N=132 peeled (33 vectors + 2 slots): 9 threads across a row");
        m = bwd(4, 1 << 16, 132, 136, base, dx, 136, &a);
        expect(m == lse::kBwdVector && a.block.x == 9 && !a.small,
               "f32 N=132 on boundaries (33 vectors): 9 threads across a row");
    }

    // Value over a non-last dimension: one warp per column tile up to R = 64,
    // 2 or 4 warps sharing a tile beyond, row splits filling one wave.
    {
        // Column-kernel CTAs per SM: 8 (f32; 4 warps per CTA), 4 with 8-warp
        // tiles; 16-bit: 6 one-warp tiles, 7 shared, 3 with 8 warps.
        auto occ = [](int dt, bool, int wt) -> int {
            if (dt == LSE_F32) return wt == 8 ? 4 : 8;
            return wt == 1 ? 6 : (wt == 8 ? 3 : 7);
        };
        auto cols = [&](lse_dtype dt, int64_t A, int64_t R, int64_t C, const void* x,
                        const lse_plan* req, lse_status* st) {
            lse_plan q;
            std::memset(&q, 0, sizeof q);
            *st = plan_columns(x, dt, A, R, C, R * C, C, 152, occ, req, &q);
            return q;
        };
        lse_status cst;
        lse_plan q = cols(LSE_F32, 512, 64, 1024, kAligned, nullptr, &cst);
        expect(cst == LSE_OK && q.path == LSE_PATH_COLUMNS_WARP && q.splits == 1 && q.grid == 1024 &&
                   q.threads == 128 && q.vector_bytes == 16,
               "[512, 64, 1024] f32: a warp per tile, no split, 1024 CTAs");
        q = cols(LSE_F32, 1, 8192, 16384, kAligned, nullptr, &cst);
        expect(cst == LSE_OK && q.path == LSE_PATH_COLUMNS_CTA && q.lanes_per_row == 4 &&
                   q.splits == 9 && q.segment_slots == 911 && q.grid == 1152 && q.launches == 2,
               "[1, 8192, 16384] f32: 4 warps per tile, 9 splits of 911 rows");
        q = cols(LSE_F32, 64, 100, 1000, kAligned, nullptr, &cst);
        expect(cst == LSE_OK && q.lanes_per_row == 2, "R = 100: 2 warps per tile");
        q = cols(LSE_F32, 512, 64, 1023, kAligned, nullptr, &cst);
        expect(cst == LSE_OK && q.vector_bytes == 1, "C = 1023: one element per lane");
        // Narrow C: one-warp tiles of 16 lanes, two per warp, at any R.
        q = cols(LSE_BF16, 8192, 128, 128, kAligned, nullptr, &cst);
        expect(cst == LSE_OK && q.path == LSE_PATH_COLUMNS_WARP && q.lanes_per_row == 1,
               "[8192, 128, 128] bf16 (half the lanes of a 32-lane tile idle): a warp per two tiles");
        expect(lse::cols_lanes_per_tile(LSE_BF16, true, 128, 1) == 16 &&
                   lse::cols_lanes_per_tile(LSE_BF16, true, 256, 1) == 32 &&
                   lse::cols_lanes_per_tile(LSE_F32, true, 128, 1) == 32 &&
                   lse::cols_lanes_per_tile(LSE_F32, true, 64, 1) == 16 &&
                   lse::cols_lanes_per_tile(LSE_BF16, true, 128, 2) == 32,
               "lanes per column tile");
        // 8-lane tiles where a 16-lane tile would leave a quarter idle too.
        expect(lse::cols_lanes_per_tile(LSE_BF16, true, 64, 1) == 8 &&
                   lse::cols_lanes_per_tile(LSE_BF16, true, 192, 1) == 8 &&
                   lse::cols_lanes_per_tile(LSE_BF16, true, 384, 1) == 16 &&
                   lse::cols_lanes_per_tile(LSE_F32, true, 32, 1) == 8 &&
                   lse::cols_lanes_per_tile(LSE_F32, false, 8, 1) == 8 &&
                   lse::cols_lanes_per_tile(LSE_BF16, true, 64, 4) == 32,
               "8-lane column tiles");
        // Narrow C over long reductions: f32 shares a narrow tile among 4 warps,
        // 16-bit keeps one warp per tile.
        q = cols(LSE_F32, 4096, 256, 64, kAligned, nullptr, &cst);
        expect(cst == LSE_OK && q.path == LSE_PATH_COLUMNS_CTA && q.lanes_per_row == 4 && q.splits == 1,
               "[4096, 256, 64] f32: 4 warps per 16-lane tile");
        q = cols(LSE_BF16, 8192, 256, 64, kAligned, nullptr, &cst);
        expect(cst == LSE_OK && q.path == LSE_PATH_COLUMNS_WARP && q.lanes_per_row == 1,
               "[8192, 256, 64] bf16: one warp per 8-lane tile");
        q = cols(LSE_BF16, 16384, 64, 64, kAligned, nullptr, &cst);
        expect(cst == LSE_OK && q.path == LSE_PATH_COLUMNS_WARP && q.lanes_per_row == 1 && q.splits == 1 &&
                   q.grid == 16384 / 16,
               "[16384, 64, 64] bf16: 8-lane tiles, four per warp, 16 per CTA");
        // Short reductions: a thread per 16-byte column vector, R <= 8.
        q = cols(LSE_F32, 1024, 2, 1024, kAligned, nullptr, &cst);
        expect(cst == LSE_OK && q.path == LSE_PATH_COLUMNS_SHORT && q.splits == 1 && q.threads == 256 &&
                   q.segment_slots == 2 && q.grid == 1024 && q.launches == 1,
               "[1024, 2, 1024] f32: short reduction, 1024 CTAs");
        q = cols(LSE_BF16, 1 << 20, 8, 64, kAligned, nullptr, &cst);
        expect(cst == LSE_OK && q.path == LSE_PATH_COLUMNS_SHORT && q.grid == 152 * 32,
               "[1M, 8, 64] bf16: short reduction, 4 waves of 8 CTAs per SM");
        q = cols(LSE_F32, 1024, 9, 1024, kAligned, nullptr, &cst);
        expect(cst == LSE_OK && q.path == LSE_PATH_COLUMNS_WARP, "R = 9: column tiles");
        q = cols(LSE_F32, 512, 4, 1023, kAligned, nullptr, &cst);
        expect(cst == LSE_OK && q.path == LSE_PATH_COLUMNS_WARP && q.vector_bytes == 1,
               "C = 1023 (element layout): column tiles");
        {
            lse_plan r2;
            std::memset(&r2, 0, sizeof r2);
            r2.splits = 2;
            q = cols(LSE_F32, 1024, 4, 1024, kAligned, &r2, &cst);
            expect(cst == LSE_OK && q.path == LSE_PATH_COLUMNS_WARP && q.splits == 2,
                   "R = 4 with 2 splits asked: column tiles");
            std::memset(&r2, 0, sizeof r2);
            r2.path = LSE_PATH_COLUMNS_SHORT;
            q = cols(LSE_F32, 1024, 4, 1024, kAligned, &r2, &cst);
            expect(cst == LSE_OK && q.path == LSE_PATH_COLUMNS_SHORT, "short path forced");
            q = cols(LSE_F32, 1024, 9, 1024, kAligned, &r2, &cst);
            expect(cst == LSE_ERR_INVALID_ARG, "short path forced on R = 9: invalid");
            q = cols(LSE_F32, 512, 4, 1023, kAligned, &r2, &cst);
            expect(cst == LSE_ERR_INVALID_ARG, "short path forced on an element layout: invalid");
            r2.splits = 2;
            q = cols(LSE_F32, 1024, 4, 1024, kAligned, &r2, &cst);
            expect(cst == LSE_ERR_INVALID_ARG, "short path forced with splits: invalid");
        }
        q = cols(LSE_F32, 4096, 128, 128, kAligned, nullptr, &cst);
        expect(cst == LSE_OK && q.lanes_per_row == 2, "[4096, 128, 128] f32 (full 32-lane tiles): 2 warps per tile");
        lse_plan r;
        std::memset(&r, 0, sizeof r);
        r.vector_bytes = 16;
        cols(LSE_F32, 512, 64, 1023, kAligned, &r, &cst);
        expect(cst == LSE_ERR_INVALID_ARG, "vectors forced on C = 1023: invalid");
        std::memset(&r, 0, sizeof r);
        r.path = LSE_PATH_COLUMNS_WARP;
        r.lanes_per_row = 2;
        cols(LSE_F32, 512, 64, 1024, kAligned, &r, &cst);
        expect(cst == LSE_ERR_INVALID_ARG, "one-warp path with 2 warps per tile: invalid");
        std::memset(&r, 0, sizeof r);
        r.path = LSE_PATH_COLUMNS_CTA;
        q = cols(LSE_BF16, 4, 512, 4096, kAligned, &r, &cst);
        expect(cst == LSE_OK && q.lanes_per_row == 8 && q.threads == 256, "forced CTA path: 8 warps per tile");
    }

    std::printf(g_fail ? "planner: %d failures\n" : "planner: ok\n", g_fail);
    return g_fail != 0;
}
