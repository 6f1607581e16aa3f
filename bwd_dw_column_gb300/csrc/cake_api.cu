// cake_api.cu -- the C ABI: argument validation, the GB300 window table that
// picks a variant per (H, rows, weight dtype, mode), workspace layout, and
// dispatch to the kernel launchers.  Host code only.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <utility>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/cake_rmsnorm.h"
#include "cake_launch.h"

namespace cake {

// ------------------------------------------------------------ smem attributes

cudaError_t ensure_smem_attr(const void *kernel, size_t smem)
{
    static std::mutex mu;
    static std::vector<std::pair<std::pair<int, const void *>, size_t>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> g(mu);
    for (auto &d : done)
        if (d.first.first == dev && d.first.second == kernel && d.second >= smem)
            return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess)
        return e;
    for (auto &d : done)
        if (d.first.first == dev && d.first.second == kernel) {
            d.second = smem;
            return cudaSuccess;
        }
    done.push_back({{dev, kernel}, smem});
    return cudaSuccess;
}

// ------------------------------------------------------------- window table

// GB300: 152 SMs.  The CTA count is derived from this constant, never from
// the device, so the deterministic pair's partition -- and so its dw bits --
// depend on the shape alone.
constexpr int kSMs = 152;
constexpr size_t kSmemPerSM = 220 * 1024; // budget for the rings of co-resident CTAs
constexpr int kMaxStages = 16;
// CTAs in the cluster form's one cluster (the portable maximum).
constexpr int kClusterCTAs = 8;
// Backward row sets of at most this many elements (rows * H) run as one CTA.
constexpr int64_t kOneCtaElems = 24576;

enum Kind { kFwd = 0, kBwd = 1 };

// Developer override of the table, for tuning sweeps: CAKE_TUNE holds
// comma-separated key=value pairs among vpt, groups, cps, stages, rpg, form,
// cluster, onecta, half, rslices (backward) and fvpt, fgroups, fcps, fstages
// (forward).
// Unset, the table below rules.
// A different row layout (vpt) changes the reduction order and therefore the
// bits of dx / y / rstd; a different cps or groups changes the pair's
// partition and therefore the bits of the deterministic dw.
struct Tune {
    int v[2][6] = {{0, 0, 0, 0, 0, 0}, {0, 0, 0, 0, 0, 0}}; // [kind][vpt, groups, cps, stages, rpg, form+1]
    int cluster = 0;                                         // cluster form: CTAs per cluster
    int one_cta_elems = 0;                                   // backward: one CTA up to rows * H elements
    int half = -1;                                           // rows of part of a warp: 0 off
    int narrow = -1;                                         // rows of at most 128 columns: 0 at 8 columns per thread
    int rslices = 0;                                         // the pair's reduce: partial ranges per column and warp
};

static Tune parse_tune(const char *t)
{
    Tune r;
    if (!t)
        return r;
    static const char *keys[2][6] = {{"fvpt", "fgroups", "fcps", "fstages", "frpg", "fform"},
                                     {"vpt", "groups", "cps", "stages", "rpg", "form"}};
    const char *p = t;
    while (*p) {
        const char *eq = strchr(p, '=');
        if (!eq)
            break;
        const size_t klen = (size_t)(eq - p);
        const int val = atoi(eq + 1);
        for (int k = 0; k < 2; ++k)
            for (int i = 0; i < 6; ++i)
                if (strlen(keys[k][i]) == klen && strncmp(p, keys[k][i], klen) == 0)
                    r.v[k][i] = i == 5 ? val + 1 : val;
        if (klen == 7 && strncmp(p, "cluster", 7) == 0 && val >= 1 && val <= kMaxCluster)
            r.cluster = val;
        if (klen == 6 && strncmp(p, "onecta", 6) == 0 && val >= 0)
            r.one_cta_elems = val;
        if (klen == 4 && strncmp(p, "half", 4) == 0 && (val == 0 || val == 1))
            r.half = val;
        if (klen == 6 && strncmp(p, "narrow", 6) == 0 && (val == 0 || val == 1))
            r.narrow = val;
        if (klen == 7 && strncmp(p, "rslices", 7) == 0 && (val == 1 || val == 2 || val == 4 || val == 8))
            r.rslices = val;
        const char *comma = strchr(eq, ',');
        if (!comma)
            break;
        p = comma + 1;
    }
    return r;
}

static const Tune &tune()
{
    static const Tune t = parse_tune(getenv("CAKE_TUNE"));
    return t;
}

struct RowLayout {
    int vpt, W;
    int lanes; // rows of part of a warp: lanes per row (16 or 8; W 1); 0: whole warps
};

static RowLayout layout_for(int H, int vpt)
{
    const int nvec = H / 8;
    return {vpt, (nvec + 32 * vpt - 1) / (32 * vpt)};
}

// The row layout fixes which thread owns which columns and therefore the
// reduction order of every per-row sum.  It depends on H (and on whether it
// is the forward or the backward) alone, so dx, y and rstd are the same bits
// whatever else the table picks.  Both directions put rows of at most 256
// columns on part of a warp; wider rows follow the rules below.
static RowLayout row_layout(int H, Kind kind)
{
    const int forced = tune().v[kind][0];
    if (forced >= 1 && forced <= 4) {
        RowLayout l = layout_for(H, forced);
        if ((l.W + 1) * 32 <= kMaxThreadsFor(forced))
            return l;
    }
    const int nvec = H / 8;
    // rows of at most 256 columns: part of a warp per row at 16 columns per
    // thread, so that one short butterfly reduces several rows and no lane
    // idles -- 136 to 256 columns on half a warp, 72 to 128 on a quarter, at
    // most 64 on an eighth (two, four or eight rows per warp).  GB300, 16
    // against 8 columns per thread on twice the lanes: H = 64, T = 524288
    // backward pair 37.2 vs 39.3 us, forward 22.7 vs 27.0 us; H = 128, T =
    // 262144 36.9 vs 40.3 us and 21.8 vs 27.1 us.  (Rows of one warp at 8
    // columns per thread took 123 and 67 us for the backward.)
    if (nvec <= 32 && tune().half != 0) {
        if (nvec > 16)
            return {2, 1, 16};
        if (tune().narrow == 0)
            return {1, 1, nvec > 8 ? 16 : 8};
        return {2, 1, nvec > 8 ? 8 : 4};
    }
    if (nvec <= 32)
        return {1, 1};
    // rows of 264 to 1024 columns: one warp per row at the fewest vectors
    // per thread that cover it.  It has as many vector slots as 8 columns per
    // thread on that many warps, but no cross-warp barrier per row, and 16 to
    // 32 columns share each thread's per-row work (GB300, T = 65536 unless
    // noted.  Backward pair, against 8 columns per thread on 2-4 warps: H =
    // 320 39.2 vs 41.7 us, 384 39.6 vs 42.2, 512 40.8 vs 43.3, 576 49.4 vs
    // 55.9, 640 49.9 vs 56.5, 704 50.9 vs 57.4, 832 63.7 vs 69.6; T = 131072,
    // H = 640 88.3 vs 99.2, 832 113.8 vs 127.1.  Forward, against 16 columns
    // per thread on 2 warps: H = 576 27.0 vs 38.1 us, 640 28.1 vs 38.6, 768
    // 31.3 vs 39.3, 832 34.6 vs 40.1, 1024 42.1 vs 43.2)
    if (nvec <= 128)
        return {(nvec + 31) / 32, 1};
    // backward, 24 or 32 columns per thread where the row splits into W warps
    // with W dividing 12 and enough of the lanes' vectors in use: an SM then
    // holds 12 consumer warps as 12 / W row groups (or, W = 1, as three CTAs
    // of four groups), so each thread's per-row work -- the row sums, their
    // barrier, the rstd and the dx scale -- is shared by 24 or 32 columns
    // instead of 8.  "Enough" is 3/4, or 7/8 where 8 columns per thread
    // still fit four row groups in a CTA (W <= 6): a row's time is that of
    // its busiest warp, so idle lanes cost their share of the bytes.  The
    // wider vector wins a tie.  GB300, T = 65536, deterministic pair against
    // 8 columns per thread: H = 768 0.85 vs 0.77 of the copy peak, 1024 0.86
    // vs 0.81, 1792 0.86 vs 0.84, 2048 0.91 vs 0.87, 2304 0.91 vs 0.77, 2560
    // 0.90 vs 0.80, 3072 0.93 vs 0.88, 3584 0.90 vs 0.80, 4096 0.94 vs 0.88,
    // 4608 0.93 vs 0.92, 5376 0.92 vs 0.80, 6144 0.96 vs 0.84; H = 1152 and
    // 1280 (3/4 and 5/6 of the lanes at 24 columns) ran 0.69 and 0.78 against
    // 0.76 and 0.85, hence the 7/8.
    if (kind == kBwd) {
        const int w8 = (nvec + 31) / 32;
        const int need_num = w8 <= 6 ? 7 : 3, need_den = w8 <= 6 ? 8 : 4;
        RowLayout best{0, 0};
        int best_used = 0, best_slots = 1;
        for (int vpt = 4; vpt >= 3; --vpt) {
            const RowLayout l = layout_for(H, vpt);
            const int slots = 32 * vpt * l.W;
            if (12 % l.W != 0 || need_den * nvec < need_num * slots)
                continue;
            if ((int64_t)nvec * best_slots > (int64_t)best_used * slots) {
                best = l;
                best_used = nvec;
                best_slots = slots;
            }
        }
        if (best.vpt)
            return best;
    }
    // backward, 4096 < H <= 5376 outside the rule above: 24 columns per
    // thread on 7 warps, two CTAs per SM (GB300, T = 65536: H = 5120 0.93 of
    // the copy peak, against 0.89 with 32 columns on 5 warps)
    if (kind == kBwd && nvec > 32 * 16 && nvec <= 32 * 3 * 7)
        return layout_for(H, 3);
    if (kind == kBwd && nvec <= 32 * 24)
        return layout_for(H, 1);
    // forward: 16 columns per thread up to H = 4096, then 24 (measured on
    // GB300: H = 6144 runs 7 % faster with 24 than with 16)
    for (int vpt = nvec <= 512 ? 2 : 3; vpt <= 4; ++vpt) {
        RowLayout l = layout_for(H, vpt);
        if ((l.W + 1) * 32 <= kMaxThreadsFor(vpt))
            return l;
    }
    return layout_for(H, 4);
}

struct Plan {
    RowLayout rl;
    int groups, rpg, stages, ctas_per_sm, ctas;
    size_t lo_bytes;
    uint32_t rows_per_cta;
    size_t smem;
    int single, dwm;
};

static size_t ring_smem(int ntens, int rows_per_stage, int H, int stages, size_t lo_bytes)
{
    return (size_t)kMiscBytes + weight_smem_bytes(H) + lo_bytes + (size_t)stages * ntens * rows_per_stage * H * 2;
}

// Shared memory the blocked dw form keeps its per-thread compensated pair
// in: the low parts, 8 floats per vector per consumer thread, and with 8
// columns per thread the high parts as well.
static size_t lo_smem(Kind kind, int dwm, const RowLayout &rl, int groups)
{
    if (kind != kBwd || dwm != CAKE_DW_BLOCKED)
        return 0;
    const size_t n = (size_t)groups * rl.W * 32 * rl.vpt * 32 * (rl.vpt == 1 ? 2 : 1);
    return (n + 1023) & ~size_t(1023);
}

// Registers per thread of each row kernel as compiled for sm_103a (ptxas
// -v), by kind and VPT; the resident-CTA count below follows from them and
// a GPU test checks it against the occupancy the runtime reports.
static int kernel_regs(Kind kind, int vpt, int rpg, int dwm, int lanes)
{
    static const int fwd[5] = {0, 52, 72, 96, 96};
    if (kind == kFwd)
        return fwd[vpt];
    if (lanes && vpt == 2)
        return dwm == CAKE_DW_PLAIN || dwm == CAKE_DW_KAHAN ? 112 : 128; // rows of half a warp
    if (lanes)
        return 72; // rows of a half or a quarter of a warp at 8 columns per thread
    if (vpt == 1 && rpg == 2)
        return 96;
    if (vpt == 1)
        return dwm == CAKE_DW_PLAIN ? 64 : 72;
    return 128;
}

static int resident_limit(Kind kind, int vpt, int rpg, int dwm, int lanes, int warps_per_cta)
{
    const int regs = (kernel_regs(kind, vpt, rpg, dwm, lanes) + 7) & ~7;
    const int by_regs = 65536 / (warps_per_cta * 32 * regs);
    const int by_warps = 64 / warps_per_cta;
    return by_regs < by_warps ? by_regs : by_warps;
}

// Per-H CTA shape: row groups (rows in flight) per CTA and CTAs per SM.
// Backward rows of several warps: one CTA per SM holding as many row groups
// as fit its consumer warps (measured on GB300 at T = 65536: H = 1536 runs
// 17 % faster as 4 groups in one CTA than as 3 CTAs of one group, H = 2048
// 7 % faster as 3 groups, and the fewer CTA partials shorten the dw
// reduction).  Otherwise about 8 consumer warps per CTA, then as many CTAs
// per SM as the register file holds (at most 3).
static void cta_shape(const RowLayout &rl, Kind kind, int rpg, int dwm, int ntens, uint32_t rows, bool one_cta,
                      int &groups, int &ctas_per_sm)
{
    const int W = rl.W;
    const int max_warps = (rpg == 2 && rl.vpt == 1 && !rl.lanes ? kMaxThreadsR2 : kMaxThreadsFor(rl.vpt)) / 32 - 1; // consumer warps per CTA
    if (kind == kBwd && W > 1)
        groups = max_warps / W > 1 ? max_warps / W : 1;
    else if (kind == kBwd && rl.vpt > 1)
        groups = 4; // rows of one warp at 24 / 32 columns: three CTAs of four groups per SM
    else if (kind == kFwd && ntens == 1 && rl.vpt == 2 && W > 1)
        groups = max_warps / W > 1 ? max_warps / W : 1; // plain forward: see the cap below
    else
        groups = W >= 8 ? 1 : 8 / W;
    // backward rows of several warps, at most two per SM and more than one
    // CTA's worth: two row groups per CTA, so that more CTAs (and SMs) share
    // the rows (GB300, ncu spans of the pair at T = 64 and 256: H = 1536 9.4
    // and 9.8 us against 10.1 and 10.6 us with six groups; H = 4096 10.7 and
    // 12.1 us against 11.5 and 12.4 us with three; from T = 1024, and for
    // rows of one warp, fewer groups cost time)
    if (kind == kBwd && W > 1 && groups > 2 && !one_cta && rows <= (uint32_t)(kSMs * 2 * rpg))
        groups = 2;
    const Tune &t = tune();
    if (t.v[kind][1] > 0)
        groups = t.v[kind][1];
    while (groups * W > max_warps && groups > 1)
        --groups;
    if (W > 1 && groups > kMaxRowGroupBarriers) // one named barrier per group
        groups = kMaxRowGroupBarriers;
    ctas_per_sm = resident_limit(kind, rl.vpt, rpg, dwm, rl.lanes, groups * W + 1);
    // at most 3 resident CTAs; the forward's warp-per-row layout takes 4,
    // and its 4-warps-per-row layout runs best at 2 (GB300 measurements)
    int cap = 3;
    if (kind == kFwd && W == 1)
        cap = 4;
    else if (kind == kFwd && W > 1 && W <= 4)
        cap = 2;
    // plain forward at 16 columns per thread (H = 1024 .. 4096): two CTAs of
    // about 12 consumer warps (GB300, T = 65536: H = 1024 15 %, H = 1536 22 %,
    // H = 2048 2 %, H = 4096 4 % faster than the earlier 8-warp CTAs);
    // residual forward at 24 columns on 8 warps (H = 6144): one CTA per SM
    // (5 % faster)
    if (kind == kFwd && ntens == 1 && rl.vpt == 2 && W > 1)
        cap = 2;
    if (kind == kFwd && ntens == 2 && rl.vpt == 3 && W == 8)
        cap = 1;
    if (ctas_per_sm > cap)
        ctas_per_sm = cap;
    if (ctas_per_sm < 1)
        ctas_per_sm = 1;
    if (t.v[kind][2] > 0)
        ctas_per_sm = t.v[kind][2];
}

// Rows a row group owns per stage: two (interleaved, one barrier for both)
// where a row is so wide that only one group of its warps fits a CTA (13 to
// 16 warps: H = 3080 .. 4096), so that two rows are in flight per SM instead
// of one (GB300, T = 65536: H = 3584 det 16 %, H = 4096 19 % faster).
// Otherwise one, and more groups per CTA instead.
static int rows_per_group(const RowLayout &rl, Kind kind)
{
    if (rl.lanes)
        return 32 / rl.lanes; // a warp's rows of part of a warp
    int rpg = 1;
    const int one_row_groups = (kMaxThreadsFor(rl.vpt) / 32 - 1) / rl.W;
    if (kind == kBwd && rl.W > 1 && one_row_groups < 2)
        rpg = 2;
    const int forced = tune().v[kind][4];
    if (forced == 1 || forced == 2)
        rpg = forced;
    if (kind != kBwd || rl.vpt != 1 || rl.W > kMaxThreadsR2 / 32 - 1)
        rpg = 1;
    return rpg;
}

static Plan make_plan(int H, uint32_t rows, int ntens, Kind kind, int single, int dwm)
{
    Plan p;
    p.rl = row_layout(H, kind);
    p.rpg = rows_per_group(p.rl, kind);
    const int64_t one_cta = tune().one_cta_elems > 0 ? tune().one_cta_elems : kOneCtaElems;
    const bool one_cta_rows = kind == kBwd && (int64_t)rows * H <= one_cta;
    cta_shape(p.rl, kind, p.rpg, dwm, ntens, rows, one_cta_rows, p.groups, p.ctas_per_sm);
    const size_t per_cta = kSmemPerSM / p.ctas_per_sm;
    const size_t stage = (size_t)ntens * p.groups * p.rpg * H * 2;
    p.lo_bytes = lo_smem(kind, dwm, p.rl, p.groups);
    const size_t fixed = (size_t)kMiscBytes + weight_smem_bytes(H) + p.lo_bytes;
    int stages = per_cta > fixed ? (int)((per_cta - fixed) / stage) : 0;
    // Fewer bytes in flight than would fit run faster in places.  Backward
    // rows of part of a warp, or of one warp at 16 or more columns per
    // thread: at most four stages (GB300: [T, 24, 256] strided per-head views
    // at T = 32768 192 us against 199-206 us with 3, 5, 6 or 8 stages;
    // [T, 4, 256] 33.3 us against 34.3-35.0 us; H = 512, T = 131072 71.9 us
    // against 73.6 us with 7 stages).  Forward rows of one warp or less: at
    // most four stages too (H = 256, T = 131072 22.3 against 23.7 us; H =
    // 512, T = 65536 22.8 against 24.0 us).  Wider forward rows keep what
    // fits: three stages won at H = 2048 and 6144 but lost 4-6 % at H = 4096
    // and on the residual route at H = 6144.
    int want = kMaxStages;
    if (kind == kBwd && p.rl.W == 1 && (p.rl.vpt >= 2 || p.rl.lanes))
        want = 4;
    if (kind == kFwd && p.rl.W == 1)
        want = 4;
    if (tune().v[kind][3] >= 2)
        want = tune().v[kind][3];
    if (want < stages)
        stages = want;
    if (stages > kMaxStages)
        stages = kMaxStages;
    if (stages < 2) { // fewer CTAs per SM so that at least two stages fit
        p.ctas_per_sm = 1;
        stages = (int)((kSmemPerSM - fixed) / stage);
        if (stages > kMaxStages)
            stages = kMaxStages;
    }
    p.stages = stages;
    p.smem = ring_smem(ntens, p.groups * p.rpg, H, stages, p.lo_bytes);
    // the backward's group-combine buffer (every group's partial) reuses the ring
    const size_t comb = fixed + (size_t)(kind == kBwd ? p.groups : 0) * H * 8;
    if (comb > p.smem)
        p.smem = comb;
    const uint32_t tile = (uint32_t)(p.groups * p.rpg);
    const uint32_t max_ctas = (uint32_t)kSMs * p.ctas_per_sm;
    uint32_t ctas = rows == 0 ? 0 : (rows + tile - 1) / tile; // at least one tile per CTA
    if (ctas > max_ctas)
        ctas = max_ctas;
    // backward over a few rows: one CTA, whose partial is dw, so the pair is
    // a single launch (GB300, event-timed: H = 256 T = 16 8.3 us against
    // 10.2 us for two CTAs and the reduce; H = 4096 T = 4 10.5 against 12.3;
    // H = 6144 T = 4 11.8 against 13.1; even at H = 1536 T = 16 and H = 256
    // T = 64, slower beyond: one SM cannot stream more rows in time)
    if (one_cta_rows && ctas > 1)
        ctas = 1;
    p.rows_per_cta = ctas ? (rows + ctas - 1) / ctas : 0;
    p.ctas = p.rows_per_cta ? (int)((rows + p.rows_per_cta - 1) / p.rows_per_cta) : 0;
    p.single = single;
    p.dwm = dwm;
    if (single == kFormCluster && rows > 0) {
        // one cluster of CTAs over all rows (at least one tile each)
        int C = tune().cluster > 0 ? tune().cluster : kClusterCTAs;
        const uint32_t by_tiles = (rows + tile - 1) / tile;
        if ((uint32_t)C > by_tiles)
            C = (int)by_tiles;
        p.rows_per_cta = (rows + C - 1) / C;
        p.ctas = (int)((rows + p.rows_per_cta - 1) / p.rows_per_cta);
        // its partial lives in the drained ring, past the group-combine buffer
        const size_t part = fixed + (size_t)(p.groups + 1) * H * 8;
        if (part > p.smem)
            p.smem = part;
    }
    return p;
}

// Mode / accumulation choice.  Deterministic: the pair.  Non-deterministic
// mode may run a single kernel -- FP64 column accumulation in L2 (1), the
// tree (2) or the cooperative grid form (3) -- but the table picks one only
// where it beats the pair, and on GB300 none does at any measured shape: the
// pair's reduce, launched as a programmatic dependent of the main kernel,
// adds 2-5 us after it, while the single kernels' tails (the last CTA's
// finalise behind the L2 atomics, or the grid barrier) add 4-27 us (T =
// 32768 .. 131072, H = 256 .. 6144).  So both modes run the pair, whose dw
// is also reproducible; CAKE_TUNE=form=N or force_single selects a single
// kernel.  Per-thread accumulation: the plain FP32 sum, the blocked form
// (plain FP32 sums over 16 rows folded into a compensated pair whose low
// parts live in shared memory, which costs little more than the plain sum),
// Kahan, or TwoSum, by the accuracy windows below.
//
// Accuracy windows of the per-thread sums, by the rows each column sums
// (T * nh): the cheapest form whose worst dw element stayed within 0.85 of
// the budget (the pages' margin) over the accuracy protocol -- three input
// families, x and dy ~ N(0, 1) -- on GB300:
//   rows <= 2048       plain FP32 (a thread sums a handful of rows);
//   rows <= 131072     blocked: 0.81 worst over 1440 inputs at H 4096 / 5120,
//                      T 4096 .. 131072; 0.49 at 131072 rows of 256;
//   rows <= 2^20       Kahan: blocked passes 0.85 beyond 131072 rows (0.88 at
//                      T 262144, 1.15 at T 524288, 1.12 at 786432 rows of
//                      256), Kahan stays at 0.32 - 0.39 up to 786432 rows;
//   above              TwoSum (0.0006 at every measured size).
// Costs against blocked, same shapes: Kahan 0.6 - 3 % (7 % at H 5120), TwoSum
// 4 - 28 %.
static void pick_variant(uint32_t rows, int deterministic, int &single, int &dwm)
{
    (void)deterministic;
    single = kFormPair;
    if (rows <= 2048)
        dwm = CAKE_DW_PLAIN;
    else if (rows <= 131072)
        dwm = CAKE_DW_BLOCKED;
    else if (rows <= (1u << 20))
        dwm = CAKE_DW_KAHAN;
    else
        dwm = CAKE_DW_TWOSUM;
}

// Partial ranges per column per warp of the fixed-order reduce: doubled
// while the grid stays within one CTA per SM, or while a lane would sum more
// than 32 partials.  Fewer, longer-running CTAs beat a grid of several per
// SM, even with three rounds of loads per lane (GB300, the pair's reduce
// after its main kernel: H = 5120, 304 partials, 3.9 us with 160 CTAs
// against 5.5 us with 640; H = 4096 and 6144 at 152 partials 3.0 and 3.4 us
// with 128 and 192 CTAs against 5.2 and 5.8 us with 512 and 768; H = 2048
// 2.1 us at 128 CTAs, 3.1 us at 64 and 256).
static int reduce_slices(int H, int P)
{
    if (tune().rslices > 0)
        return tune().rslices;
    int S = 1;
    while (S < 8 && ((H + 16 / S - 1) / (16 / S) <= kSMs || (P + 16 * S - 1) / (16 * S) > 32))
        S *= 2;
    return S;
}

// ---------------------------------------------------------- workspace layout

// Header words (u32): [0] the single kernel's arrival counter; [1 .. 1 + 1 +
// kTreeMaxGroups] the tree form's counters; [kGridWords, +1] the grid form's
// barrier counter and generation.
constexpr size_t kWsHeader = 512;
constexpr int kTreeMaxGroups = 62;
constexpr int kGridWords = 64;
constexpr int kAccBanks = kMaxAccBanks; // copies of the single kernel's FP64 accumulators

static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

static size_t ws_acc_off() { return kWsHeader; }
static size_t ws_part_off(int H) { return align256(kWsHeader + (size_t)kAccBanks * H * 8); }
static size_t ws_size(int H, int ctas, int need_partials)
{
    return ws_part_off(H) + (need_partials ? (size_t)ctas * H * 8 : 0);
}
static int tree_groups(int ctas) { return (ctas + kTreeGroup - 1) / kTreeGroup; }
static size_t ws_tree_off(int H, int ctas) { return align256(ws_size(H, ctas, 1)); }
// Bytes each form needs: the atomic single kernel its counter and one bank,
// the pair its partials, the tree its partials and the group totals.
static size_t ws_need(int form, int H, int ctas)
{
    if (form == kFormCluster)
        return 0; // the partials stay in the cluster's shared memory
    if (form == kFormAtomic)
        return kWsHeader + (size_t)H * 8;
    if (form == kFormTree)
        return ws_tree_off(H, ctas) + (size_t)tree_groups(ctas) * H * 8;
    return ws_size(H, ctas, 1);
}

} // namespace cake

using namespace cake;

// ------------------------------------------------------------- validation

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cake_status check_shape(const cake_shape *s, uint32_t *rows)
{
    if (!s || s->tokens < 0 || s->heads < 1 || s->hidden < 1)
        return CAKE_ERR_INVALID;
    if (s->hidden % 8 != 0 || s->hidden > CAKE_MAX_HIDDEN)
        return CAKE_ERR_UNSUPPORTED;
    const int64_t r = s->tokens * s->heads;
    if (s->tokens > 0 && r / s->tokens != s->heads)
        return CAKE_ERR_UNSUPPORTED;
    if (r >= (int64_t(1) << 31))
        return CAKE_ERR_UNSUPPORTED;
    *rows = (uint32_t)r;
    return CAKE_OK;
}

// Activation tensor: non-null, 16-byte aligned base, strides multiples of 8
// elements (16 bytes) and non-negative.
cake_status check_tensor(const cake_tensor *t, const cake_shape *s)
{
    if (!t || !t->data)
        return CAKE_ERR_INVALID;
    if (t->stride_token < 0 || t->stride_head < 0)
        return CAKE_ERR_UNSUPPORTED;
    if (!aligned16(t->data) || t->stride_token % 8 != 0 ||
        (s->heads > 1 && t->stride_head % 8 != 0))
        return CAKE_ERR_UNSUPPORTED;
    if (s->tokens > 1 && t->stride_token < (s->heads > 1 ? 0 : s->hidden))
        return CAKE_ERR_UNSUPPORTED;
    if (s->heads > 1 && t->stride_head < s->hidden)
        return CAKE_ERR_UNSUPPORTED;
    return CAKE_OK;
}

// An output tensor: as check_tensor, and no two of its rows overlap (a
// kernel writes every row once, so rows that share memory would race).  The
// dimensions with more than one index, in ascending stride order, must each
// step past everything the smaller ones span.
cake_status check_out_tensor(const cake_tensor *t, const cake_shape *s)
{
    cake_status st = check_tensor(t, s);
    if (st != CAKE_OK)
        return st;
    int64_t dims[2][2] = {{s->tokens, t->stride_token}, {s->heads, t->stride_head}};
    if (dims[0][1] > dims[1][1]) {
        std::swap(dims[0][0], dims[1][0]);
        std::swap(dims[0][1], dims[1][1]);
    }
    int64_t span = s->hidden; // elements one index of the dimensions seen so far covers
    for (auto &d : dims) {
        if (d[0] <= 1)
            continue;
        if (d[1] < span)
            return CAKE_ERR_INVALID;
        span = (d[0] - 1) * d[1] + span;
    }
    return CAKE_OK;
}

// Byte range [lo, hi) a view's rows touch (strides are non-negative).
std::pair<uintptr_t, uintptr_t> extent(const cake_tensor *t, const cake_shape *s)
{
    const uintptr_t lo = reinterpret_cast<uintptr_t>(t->data);
    const int64_t last = (s->tokens - 1) * t->stride_token + (s->heads > 1 ? (s->heads - 1) * t->stride_head : 0);
    return {lo, lo + (uintptr_t)(2 * (last + s->hidden))};
}

bool overlap(const cake_tensor *a, const cake_tensor *b, const cake_shape *s)
{
    if (!a || !a->data || !b || !b->data)
        return false;
    const auto ea = extent(a, s), eb = extent(b, s);
    return ea.first < eb.second && eb.first < ea.second;
}

bool same_view(const cake_tensor *a, const cake_tensor *b, const cake_shape *s)
{
    return a->data == b->data && (s->tokens <= 1 || a->stride_token == b->stride_token) &&
           (s->heads <= 1 || a->stride_head == b->stride_head);
}

RowView make_view(const cake_tensor *t, const cake_shape *s)
{
    RowView v{};
    if (!t || !t->data)
        return v;
    v.base = static_cast<const uint16_t *>(t->data);
    v.st = t->stride_token;
    v.sh = s->heads > 1 ? t->stride_head : 0;
    if (s->heads == 1) {
        v.uniform = 1;
        v.row_stride = t->stride_token;
    } else if (t->stride_token == s->heads * t->stride_head) {
        v.uniform = 1;
        v.row_stride = t->stride_head;
    } else if (s->tokens == 1) {
        v.uniform = 1;
        v.row_stride = t->stride_head;
    }
    v.dense = v.uniform && v.row_stride == s->hidden;
    return v;
}

cake_status cuda_status(cudaError_t e)
{
    return e == cudaSuccess ? CAKE_OK : CAKE_ERR_CUDA;
}

Layout make_layout(const Plan &p, int H, uint32_t rows, uint32_t nh, int ntens)
{
    Layout L;
    L.H = H;
    L.nvec = H / 8;
    L.warps_per_row = p.rl.W;
    L.groups = p.groups;
    L.rows_per_group = p.rpg;
    L.lanes_per_row = p.rl.lanes ? p.rl.lanes : 32;
    L.stages = p.stages;
    L.lo_bytes = (int)p.lo_bytes;
    L.ntens = ntens;
    L.rows = rows;
    L.nh = nh;
    L.rows_per_cta = p.rows_per_cta;
    L.inv_h = 1.0f / (float)H;
    return L;
}

void fill_variant(const Plan &p, cake_variant *out)
{
    out->single = p.single;
    out->dw_accum = p.dwm;
    out->vec_per_thread = p.rl.vpt;
    out->warps_per_row = p.rl.W;
    out->row_groups = p.groups;
    out->rows_per_group = p.rpg;
    out->stages = p.stages;
    out->ctas = p.ctas;
    out->rows_per_cta = p.rows_per_cta;
    out->smem_bytes = p.smem;
    out->lanes_per_row = p.rl.lanes ? p.rl.lanes : 32;
}

cake_status select_plan(const cake_shape *shape, int deterministic, int has_dh, int force_single,
                        int force_accum, Plan *plan, uint32_t *rows)
{
    cake_status st = check_shape(shape, rows);
    if (st != CAKE_OK)
        return st;
    if (force_single > kFormCluster || force_accum > CAKE_DW_KAHAN)
        return CAKE_ERR_INVALID;
    if (deterministic && force_single == kFormAtomic)
        return CAKE_ERR_INVALID;
    int single, dwm;
    pick_variant(*rows, deterministic, single, dwm);
    if (tune().v[kBwd][5] > 0 && (tune().v[kBwd][5] - 1 != kFormAtomic || !deterministic))
        single = tune().v[kBwd][5] - 1;
    if (force_single >= 0)
        single = force_single;
    if (force_accum >= 0)
        dwm = force_accum;
    *plan = make_plan((int)shape->hidden, *rows, has_dh ? 3 : 2, kBwd, single, dwm);
    // the tree form is built for 8 or 16 columns per thread
    if (plan->single == kFormTree &&
        (plan->rl.vpt > 2 || (plan->rl.vpt == 1 && plan->rpg != 1 && !plan->rl.lanes) ||
         tree_groups(plan->ctas) > kTreeMaxGroups))
        return CAKE_ERR_UNSUPPORTED;
    return CAKE_OK;
}

enum Phase { kWhole = 0, kMainOnly = 1 };

cake_status run_bwd(const cake_shape *shape, const cake_tensor *dy, const cake_tensor *x,
                    const float *rstd, const void *w, cake_dtype w_dtype, const cake_tensor *dh,
                    const cake_tensor *dx, float *dw, void *workspace, size_t workspace_bytes,
                    int deterministic, int force_single, int force_accum, cake_stream_t stream,
                    Phase phase = kWhole, uint64_t wait_ns = kWaitLimitNs, int grid_extra = 0)
{
    uint32_t rows = 0;
    const int has_dh = dh && dh->data;
    Plan plan;
    cake_status st = select_plan(shape, deterministic, has_dh, force_single, force_accum, &plan, &rows);
    if (st != CAKE_OK)
        return st;
    if (w_dtype != CAKE_BF16 && w_dtype != CAKE_FP32)
        return CAKE_ERR_INVALID;
    if (!dw || !w)
        return CAKE_ERR_INVALID;
    if (!aligned16(w) || !aligned16(dw))
        return CAKE_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int H = (int)shape->hidden;
    if (rows == 0)
        return cuda_status(cudaMemsetAsync(dw, 0, (size_t)H * sizeof(float), s));
    if (!rstd)
        return CAKE_ERR_INVALID;
    if ((reinterpret_cast<uintptr_t>(rstd) & 3u) != 0)
        return CAKE_ERR_UNSUPPORTED;
    if ((st = check_tensor(dy, shape)) != CAKE_OK || (st = check_tensor(x, shape)) != CAKE_OK ||
        (st = check_out_tensor(dx, shape)) != CAKE_OK)
        return st;
    if (has_dh && (st = check_tensor(dh, shape)) != CAKE_OK)
        return st;
    // dx is written while later rows of dy, x and dh are still being read
    if (overlap(dx, dy, shape) || overlap(dx, x, shape) || (has_dh && overlap(dx, dh, shape)))
        return CAKE_ERR_INVALID;
    const size_t need = ws_need(plan.single, H, plan.ctas);
    if (need > 0 && (!workspace || workspace_bytes < need))
        return CAKE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return CAKE_ERR_UNSUPPORTED;

    BwdParams p{};
    p.L = make_layout(plan, H, rows, (uint32_t)shape->heads, has_dh ? 3 : 2);
    p.x = make_view(x, shape);
    p.dy = make_view(dy, shape);
    p.dh = make_view(has_dh ? dh : nullptr, shape);
    p.rstd = rstd;
    p.w = w;
    p.w_f32 = w_dtype == CAKE_FP32;
    RowView dxv = make_view(dx, shape);
    p.dx = static_cast<uint16_t *>(dx->data);
    p.dx_st = dxv.st;
    p.dx_sh = dxv.sh;
    p.dx_row_stride = dxv.row_stride;
    p.dx_uniform = dxv.uniform;
    p.dw = dw;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    if (ws) { // (the cluster form uses none of it)
        p.arrivals = reinterpret_cast<unsigned int *>(ws);
        p.acc = reinterpret_cast<double *>(ws + ws_acc_off());
        p.partials = reinterpret_cast<float2 *>(ws + ws_part_off(H));
        p.tree_cnt = reinterpret_cast<unsigned int *>(ws) + 1;
        p.group_totals = reinterpret_cast<float2 *>(ws + ws_tree_off(H, plan.ctas));
        p.grid_cnt = reinterpret_cast<unsigned int *>(ws) + kGridWords;
        p.grid_gen = reinterpret_cast<unsigned int *>(ws) + kGridWords + 1;
    }
    // the accumulator banks that fit the given workspace (the built-in
    // scratch of the allocation-free entry point may hold fewer than 8)
    {
        const size_t room = workspace_bytes > kWsHeader ? (workspace_bytes - kWsHeader) / ((size_t)H * 8) : 0;
        p.banks = room >= (size_t)kAccBanks ? kAccBanks : (int)(room > 0 ? room : 1);
        // CTA b adds into bank b % banks: more banks than CTAs would only
        // lengthen the last CTA's finalise
        if (plan.ctas > 0 && p.banks > plan.ctas)
            p.banks = plan.ctas;
    }
    p.block_rows = 16;
    p.status = nullptr;
    p.wait_ns = wait_ns;
    p.grid_extra = grid_extra;
    p.cluster = plan.single == kFormCluster ? plan.ctas : 0;
    // a pair of one CTA writes dw from the main kernel (same bits as the
    // reduce of its single partial); the separate halves keep the partial
    p.direct_dw = plan.single == kFormPair && plan.ctas == 1 && phase == kWhole;
    cudaError_t e = launch_bwd_rows(p, plan.rl.vpt, plan.single, plan.dwm, plan.ctas, plan.smem, s);
    if (e != cudaSuccess || plan.single != kFormPair || phase == kMainOnly || p.direct_dw)
        return cuda_status(e);
    ReduceParams rp{p.partials, plan.ctas, H, dw, reduce_slices(H, plan.ctas)};
    return cuda_status(launch_dw_reduce(rp, s));
}

// ------------------------------------------------------- from host buffers
//
// The backward over rows that live in host memory: the rows go in chunks, and
// the copy of chunk c + 1 to the device, the main kernel of chunk c and the
// copy of chunk c - 1's dx back overlap on three streams (the caller's for the
// kernels, two of the library's for the copies).  Every chunk's CTA partials
// stay in the staging memory and one fixed-order reduce over all of them gives
// dw, so dw is reproducible for a given shape and chunk count.

constexpr int kHostSlots = 3;       // staging slots the chunks rotate through
constexpr int kHostMaxChunks = 64;
constexpr int kHostMaxDevices = 64;

struct HostChunking {
    int chunks, slots;
    uint32_t rows_c, rows_last;  // rows of a full chunk and of the last one
    Plan full, last;
    size_t off_x, off_dy, off_dh, off_rstd, off_dx, slot_bytes; // within a slot
    size_t off_w, off_dw, off_part, total;
};

bool host_chunking(int H, uint32_t rows, int has_dh, int w_elem_bytes, int chunks, HostChunking *c)
{
    if (chunks < 1 || chunks > kHostMaxChunks || rows == 0)
        return false;
    const uint32_t k = (uint32_t)chunks < rows ? (uint32_t)chunks : rows;
    c->rows_c = (rows + k - 1) / k;
    c->chunks = (int)((rows + c->rows_c - 1) / c->rows_c); // every chunk holds rows
    c->rows_last = rows - (uint32_t)(c->chunks - 1) * c->rows_c;
    c->slots = c->chunks < kHostSlots ? c->chunks : kHostSlots;
    // the accumulation form follows the rows every column sums in all
    int single, dwm;
    pick_variant(rows, 1, single, dwm);
    const int ntens = has_dh ? 3 : 2;
    c->full = make_plan(H, c->rows_c, ntens, kBwd, kFormPair, dwm);
    c->last = make_plan(H, c->rows_last, ntens, kBwd, kFormPair, dwm);
    const size_t act = align256((size_t)c->rows_c * H * 2);
    c->off_x = 0;
    c->off_dy = act;
    c->off_dh = 2 * act;
    c->off_rstd = (has_dh ? 3 : 2) * act;
    c->off_dx = c->off_rstd + align256((size_t)c->rows_c * 4);
    c->slot_bytes = c->off_dx + act;
    c->off_w = (size_t)c->slots * c->slot_bytes;
    c->off_dw = c->off_w + align256((size_t)H * w_elem_bytes);
    c->off_part = c->off_dw + align256((size_t)H * 4);
    c->total = c->off_part + (size_t)c->chunks * c->full.ctas * H * 8;
    return true;
}

// The library's two copy streams and the events that order the chunks, per
// device, created at the first call on that device and kept.
struct HostStreams {
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, end = nullptr;
    cudaEvent_t in_ready[kHostSlots] = {}, computed[kHostSlots] = {}, out_done[kHostSlots] = {};
    std::mutex mu; // one enqueue at a time per device
    bool ready = false;
};

HostStreams g_host_streams[kHostMaxDevices];
std::mutex g_host_init_mu;

cudaError_t host_streams(int dev, HostStreams **out)
{
    if (dev < 0 || dev >= kHostMaxDevices)
        return cudaErrorInvalidDevice;
    HostStreams &h = g_host_streams[dev];
    std::lock_guard<std::mutex> g(g_host_init_mu);
    if (!h.ready) {
        cudaError_t e = cudaStreamCreateWithFlags(&h.in, cudaStreamNonBlocking);
        if (e == cudaSuccess)
            e = cudaStreamCreateWithFlags(&h.out, cudaStreamNonBlocking);
        cudaEvent_t *evs[] = {&h.start, &h.end};
        for (cudaEvent_t *ev : evs)
            if (e == cudaSuccess)
                e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        for (int i = 0; i < kHostSlots && e == cudaSuccess; ++i) {
            e = cudaEventCreateWithFlags(&h.in_ready[i], cudaEventDisableTiming);
            if (e == cudaSuccess)
                e = cudaEventCreateWithFlags(&h.computed[i], cudaEventDisableTiming);
            if (e == cudaSuccess)
                e = cudaEventCreateWithFlags(&h.out_done[i], cudaEventDisableTiming);
        }
        if (e != cudaSuccess)
            return e;
        h.ready = true;
    }
    *out = &h;
    return cudaSuccess;
}

// One chunk's main kernel: rows [0, rows) of a dense staging slot, its CTA
// partials at `partials`.
cudaError_t launch_chunk_main(const Plan &plan, int H, uint32_t rows, int has_dh, const uint16_t *x,
                              const uint16_t *dy, const uint16_t *dh, const float *rstd, const void *w,
                              int w_f32, uint16_t *dx, float *dw, float2 *partials, cudaStream_t s)
{
    const cake_shape shape{rows, 1, H};
    BwdParams p{};
    p.L = make_layout(plan, H, rows, 1, has_dh ? 3 : 2);
    const cake_tensor tx{const_cast<uint16_t *>(x), H, 0}, tdy{const_cast<uint16_t *>(dy), H, 0},
        tdh{const_cast<uint16_t *>(dh), H, 0}, tdx{dx, H, 0};
    p.x = make_view(&tx, &shape);
    p.dy = make_view(&tdy, &shape);
    p.dh = make_view(has_dh ? &tdh : nullptr, &shape);
    p.rstd = rstd;
    p.w = w;
    p.w_f32 = w_f32;
    const RowView dxv = make_view(&tdx, &shape);
    p.dx = dx;
    p.dx_st = dxv.st;
    p.dx_sh = dxv.sh;
    p.dx_row_stride = dxv.row_stride;
    p.dx_uniform = dxv.uniform;
    p.dw = dw;
    p.partials = partials;
    p.banks = 1;
    p.block_rows = 16;
    p.status = nullptr;
    p.wait_ns = kWaitLimitNs;
    return launch_bwd_rows(p, plan.rl.vpt, kFormPair, plan.dwm, plan.ctas, plan.smem, s);
}

cake_status run_bwd_host(const cake_shape *shape, const void *dy, const void *x, const float *rstd,
                         const void *w, cake_dtype w_dtype, const void *dh, void *dx, float *dw, void *staging,
                         size_t staging_bytes, int chunks, cake_stream_t stream)
{
    uint32_t rows = 0;
    cake_status st = check_shape(shape, &rows);
    if (st != CAKE_OK)
        return st;
    if (w_dtype != CAKE_BF16 && w_dtype != CAKE_FP32)
        return CAKE_ERR_INVALID;
    if (chunks < 1 || chunks > kHostMaxChunks || !w || !dw)
        return CAKE_ERR_INVALID;
    const int H = (int)shape->hidden;
    if (rows == 0) {
        std::memset(dw, 0, (size_t)H * sizeof(float)); // nothing to copy: dw is zero now
        return CAKE_OK;
    }
    if (!dy || !x || !rstd || !dx)
        return CAKE_ERR_INVALID;
    const int has_dh = dh != nullptr;
    const int wb = w_dtype == CAKE_FP32 ? 4 : 2;
    HostChunking c;
    if (!host_chunking(H, rows, has_dh, wb, chunks, &c))
        return CAKE_ERR_INVALID;
    if (!staging || staging_bytes < c.total)
        return CAKE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(staging) & 255u) != 0)
        return CAKE_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int dev = -1, sdev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaStreamGetDevice(s, &sdev) != cudaSuccess)
        return CAKE_ERR_CUDA;
    if (sdev != dev)
        return CAKE_ERR_INVALID;
    HostStreams *hs = nullptr;
    if (host_streams(dev, &hs) != cudaSuccess)
        return CAKE_ERR_CUDA;
    std::lock_guard<std::mutex> g(hs->mu);

    uint8_t *base = static_cast<uint8_t *>(staging);
    float2 *part = reinterpret_cast<float2 *>(base + c.off_part);
    float *dw_dev = reinterpret_cast<float *>(base + c.off_dw);
    const int P = c.full.ctas;
    const size_t row_bytes = (size_t)H * 2;
    cudaError_t e = cudaSuccess;
    auto ok = [&](cudaError_t r) {
        if (e == cudaSuccess)
            e = r;
        return e == cudaSuccess;
    };
    // everything after the caller's earlier work on `stream`
    ok(cudaEventRecord(hs->start, s));
    ok(cudaStreamWaitEvent(hs->in, hs->start, 0));
    ok(cudaStreamWaitEvent(hs->out, hs->start, 0));
    ok(cudaMemcpyAsync(base + c.off_w, w, (size_t)H * wb, cudaMemcpyHostToDevice, hs->in));
    // the last chunk may have fewer CTAs: its missing partials are zeros
    if (c.last.ctas < P)
        ok(cudaMemsetAsync(part + ((size_t)(c.chunks - 1) * P + c.last.ctas) * H, 0,
                           (size_t)(P - c.last.ctas) * H * 8, s));
    for (int k = 0; k < c.chunks && e == cudaSuccess; ++k) {
        const int slot = k % c.slots;
        const uint32_t n = k == c.chunks - 1 ? c.rows_last : c.rows_c;
        const size_t r0 = (size_t)k * c.rows_c;
        uint8_t *sb = base + (size_t)slot * c.slot_bytes;
        if (k >= c.slots)
            ok(cudaStreamWaitEvent(hs->in, hs->computed[slot], 0)); // inputs of chunk k - slots consumed
        ok(cudaMemcpyAsync(sb + c.off_x, static_cast<const uint8_t *>(x) + r0 * row_bytes, n * row_bytes,
                           cudaMemcpyHostToDevice, hs->in));
        ok(cudaMemcpyAsync(sb + c.off_dy, static_cast<const uint8_t *>(dy) + r0 * row_bytes, n * row_bytes,
                           cudaMemcpyHostToDevice, hs->in));
        if (has_dh)
            ok(cudaMemcpyAsync(sb + c.off_dh, static_cast<const uint8_t *>(dh) + r0 * row_bytes, n * row_bytes,
                               cudaMemcpyHostToDevice, hs->in));
        ok(cudaMemcpyAsync(sb + c.off_rstd, rstd + r0, (size_t)n * 4, cudaMemcpyHostToDevice, hs->in));
        ok(cudaEventRecord(hs->in_ready[slot], hs->in));
        ok(cudaStreamWaitEvent(s, hs->in_ready[slot], 0));
        if (k >= c.slots)
            ok(cudaStreamWaitEvent(s, hs->out_done[slot], 0)); // dx of chunk k - slots copied out
        ok(launch_chunk_main(k == c.chunks - 1 ? c.last : c.full, H, n, has_dh,
                             reinterpret_cast<const uint16_t *>(sb + c.off_x),
                             reinterpret_cast<const uint16_t *>(sb + c.off_dy),
                             reinterpret_cast<const uint16_t *>(sb + c.off_dh),
                             reinterpret_cast<const float *>(sb + c.off_rstd), base + c.off_w, w_dtype == CAKE_FP32,
                             reinterpret_cast<uint16_t *>(sb + c.off_dx), dw_dev, part + (size_t)k * P * H, s));
        ok(cudaEventRecord(hs->computed[slot], s));
        ok(cudaStreamWaitEvent(hs->out, hs->computed[slot], 0));
        ok(cudaMemcpyAsync(static_cast<uint8_t *>(dx) + r0 * row_bytes, sb + c.off_dx, n * row_bytes,
                           cudaMemcpyDeviceToHost, hs->out));
        ok(cudaEventRecord(hs->out_done[slot], hs->out));
    }
    // dw: every chunk's partials in chunk, then CTA, order
    if (e == cudaSuccess) {
        ReduceParams rp{part, c.chunks * P, H, dw_dev, reduce_slices(H, c.chunks * P)};
        ok(launch_dw_reduce(rp, s));
    }
    ok(cudaMemcpyAsync(dw, dw_dev, (size_t)H * 4, cudaMemcpyDeviceToHost, s));
    // later work on `stream` comes after the last copies of dx
    ok(cudaEventRecord(hs->end, hs->out));
    ok(cudaStreamWaitEvent(s, hs->end, 0));
    return cuda_status(e);
}

} // namespace

// ---------------------------------------------------------------------------
// Backward without any caller-provided scratch (cake_rmsnorm_bwd_noalloc).
//
// Some callers cannot hand the library device memory they allocated: code
// running inside a framework that owns every allocation, or a host path that
// must not call cudaMalloc (which can synchronise the device) in the middle
// of a step.  For them the single kernel's scratch -- its CTA arrival counter
// and its FP64 column accumulators -- lives in this library-owned array
// instead of a workspace.  It is loaded with the library and stays resident
// on every GPU that uses the library until the process exits.
constexpr size_t kNoAllocScratchBytes = kWsHeader + 8 * (size_t)CAKE_NOALLOC_MAX_HIDDEN;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

constexpr int kNoAllocMaxDevices = 64;

// Device address of g_noalloc_scratch for the current device.  In host code
// the array's name is only a stand-in for the symbol, not a device pointer,
// so the address is looked up once per device (with that device current)
// and cached.
cake_status noalloc_scratch(void **out)
{
    static std::mutex mu;
    static void *addr[kNoAllocMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices)
        return CAKE_ERR_CUDA;
    std::lock_guard<std::mutex> g(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p)
            return CAKE_ERR_CUDA;
        addr[dev] = p;
    }
    *out = addr[dev];
    return CAKE_OK;
}

} // namespace

extern "C" cake_status cake_rmsnorm_bwd_noalloc(const cake_shape *shape, const cake_tensor *dy,
                                                const cake_tensor *x, const float *rstd, const void *w,
                                                cake_dtype w_dtype, const cake_tensor *dh,
                                                const cake_tensor *dx, float *dw, cake_stream_t stream)
{
    if (!shape)
        return CAKE_ERR_INVALID;
    if (shape->hidden > CAKE_NOALLOC_MAX_HIDDEN)
        return CAKE_ERR_WORKSPACE; // more columns than the built-in scratch holds
    uint32_t rows = 0;
    cake_status st = check_shape(shape, &rows);
    if (st != CAKE_OK)
        return st;
    // The scratch address is looked up for the current device, so the stream
    // must belong to that device (a stream of another GPU would run the
    // kernel against the other GPU's copy of the array).
    int cur = -1, sdev = -1;
    if (cudaGetDevice(&cur) != cudaSuccess ||
        cudaStreamGetDevice(reinterpret_cast<cudaStream_t>(stream), &sdev) != cudaSuccess)
        return CAKE_ERR_CUDA;
    if (sdev != cur)
        return CAKE_ERR_INVALID;
    void *scratch = nullptr;
    if ((st = noalloc_scratch(&scratch)) != CAKE_OK)
        return st;
    // The counter and the accumulators must start at zero.  A completed call
    // leaves them zero, but clear them anyway (an asynchronous memset, no
    // allocation) so that an earlier call that stopped early cannot leak in.
    const size_t used = kNoAllocScratchBytes;
    if (rows > 0 &&
        cudaMemsetAsync(scratch, 0, used, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return CAKE_ERR_CUDA;
    return run_bwd(shape, dy, x, rstd, w, w_dtype, dh, dx, dw, scratch, kNoAllocScratchBytes, 0, 1, -1,
                   stream);
}

// ------------------------------------------------------------------- C ABI

extern "C" {

int cake_rmsnorm_abi_version(void) { return CAKE_ABI_VERSION; }

const char *cake_status_str(cake_status status)
{
    switch (status) {
    case CAKE_OK: return "ok";
    case CAKE_ERR_INVALID: return "invalid argument";
    case CAKE_ERR_UNSUPPORTED: return "unsupported shape, stride or alignment";
    case CAKE_ERR_WORKSPACE: return "workspace missing or too small";
    case CAKE_ERR_CUDA: return "CUDA runtime error";
    case CAKE_ERR_TIMEOUT: return "a kernel's bounded wait ran out";
    }
    return "unknown status";
}

cake_status cake_rmsnorm_fwd(const cake_shape *shape, const cake_tensor *x,
                             const cake_tensor *residual, const void *w, cake_dtype w_dtype,
                             float eps, const cake_tensor *y, const cake_tensor *h_new,
                             float *rstd, cake_stream_t stream)
{
    uint32_t rows = 0;
    cake_status st = check_shape(shape, &rows);
    if (st != CAKE_OK)
        return st;
    if (w_dtype != CAKE_BF16 && w_dtype != CAKE_FP32)
        return CAKE_ERR_INVALID;
    if (!(eps >= 0.0f))
        return CAKE_ERR_INVALID;
    const int has_res = residual && residual->data;
    if (rows == 0)
        return CAKE_OK;
    if (!w || !rstd)
        return CAKE_ERR_INVALID;
    if (!aligned16(w) || (reinterpret_cast<uintptr_t>(rstd) & 3u) != 0)
        return CAKE_ERR_UNSUPPORTED;
    if ((st = check_tensor(x, shape)) != CAKE_OK || (st = check_out_tensor(y, shape)) != CAKE_OK)
        return st;
    if (has_res) {
        if ((st = check_tensor(residual, shape)) != CAKE_OK || (st = check_out_tensor(h_new, shape)) != CAKE_OK)
            return st;
    } else if (h_new && h_new->data) {
        return CAKE_ERR_INVALID;
    }
    // Outputs may not share memory with each other, nor partly with an input:
    // a row is written only after it is read, so an output may be exactly an
    // input view (in place) but not straddle other rows of one.
    if (has_res && overlap(y, h_new, shape))
        return CAKE_ERR_INVALID;
    {
        const cake_tensor *outs[2] = {y, has_res ? h_new : nullptr};
        const cake_tensor *ins[2] = {x, has_res ? residual : nullptr};
        for (const cake_tensor *o : outs)
            for (const cake_tensor *i : ins)
                if (o && i && overlap(o, i, shape) && !same_view(o, i, shape))
                    return CAKE_ERR_INVALID;
    }
    const int H = (int)shape->hidden;
    const int ntens = has_res ? 2 : 1;
    Plan plan = make_plan(H, rows, ntens, kFwd, 0, 0);
    FwdParams p{};
    p.L = make_layout(plan, H, rows, (uint32_t)shape->heads, ntens);
    p.x = make_view(x, shape);
    p.res = make_view(has_res ? residual : nullptr, shape);
    p.w = w;
    p.w_f32 = w_dtype == CAKE_FP32;
    p.eps = eps;
    RowView yv = make_view(y, shape);
    p.y = static_cast<uint16_t *>(y->data);
    p.y_st = yv.st;
    p.y_sh = yv.sh;
    p.y_row_stride = yv.row_stride;
    p.y_uniform = yv.uniform;
    if (has_res) {
        RowView hv = make_view(h_new, shape);
        p.h_new = static_cast<uint16_t *>(h_new->data);
        p.hn_st = hv.st;
        p.hn_sh = hv.sh;
        p.hn_row_stride = hv.row_stride;
        p.hn_uniform = hv.uniform;
    }
    p.rstd = rstd;
    p.status = nullptr;
    p.wait_ns = kWaitLimitNs;
    return cuda_status(launch_fwd(p, plan.rl.vpt, plan.ctas, plan.smem,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

size_t cake_rmsnorm_bwd_workspace_size(const cake_shape *shape, cake_dtype w_dtype, int deterministic)
{
    (void)w_dtype;
    uint32_t rows = 0;
    if (check_shape(shape, &rows) != CAKE_OK || rows == 0)
        return 0;
    // the largest of every variant this mode may run (the table or a forced one)
    const int H = (int)shape->hidden;
    size_t need = 0;
    for (int ntens = 2; ntens <= 3; ++ntens)
        for (int dwm = CAKE_DW_PLAIN; dwm <= CAKE_DW_KAHAN; ++dwm) {
            Plan p = make_plan(H, rows, ntens, kBwd, 0, dwm);
            size_t n = ws_need(kFormTree, H, p.ctas);
            if (n > need)
                need = n;
        }
    (void)deterministic;
    return need;
}

cake_status cake_rmsnorm_bwd_workspace_init(void *workspace, size_t workspace_bytes, cake_stream_t stream)
{
    if (!workspace && workspace_bytes)
        return CAKE_ERR_INVALID;
    if (!workspace_bytes)
        return CAKE_OK;
    return cuda_status(cudaMemsetAsync(workspace, 0, workspace_bytes, reinterpret_cast<cudaStream_t>(stream)));
}

cake_status cake_rmsnorm_bwd_select(const cake_shape *shape, cake_dtype w_dtype, int deterministic,
                                    int has_dh, int force_single, int force_accum, cake_variant *out)
{
    if (!out)
        return CAKE_ERR_INVALID;
    if (w_dtype != CAKE_BF16 && w_dtype != CAKE_FP32)
        return CAKE_ERR_INVALID;
    Plan plan;
    uint32_t rows = 0;
    cake_status st = select_plan(shape, deterministic, has_dh, force_single, force_accum, &plan, &rows);
    if (st != CAKE_OK)
        return st;
    fill_variant(plan, out);
    return CAKE_OK;
}

cake_status cake_rmsnorm_bwd(const cake_shape *shape, const cake_tensor *dy, const cake_tensor *x,
                             const float *rstd, const void *w, cake_dtype w_dtype,
                             const cake_tensor *dh, const cake_tensor *dx, float *dw,
                             void *workspace, size_t workspace_bytes, int deterministic,
                             cake_stream_t stream)
{
    return run_bwd(shape, dy, x, rstd, w, w_dtype, dh, dx, dw, workspace, workspace_bytes,
                   deterministic, -1, -1, stream);
}

cake_status cake_rmsnorm_bwd_forced(const cake_shape *shape, const cake_tensor *dy,
                                    const cake_tensor *x, const float *rstd, const void *w,
                                    cake_dtype w_dtype, const cake_tensor *dh, const cake_tensor *dx,
                                    float *dw, void *workspace, size_t workspace_bytes,
                                    int deterministic, int force_single, int force_accum,
                                    cake_stream_t stream)
{
    return run_bwd(shape, dy, x, rstd, w, w_dtype, dh, dx, dw, workspace, workspace_bytes,
                   deterministic, force_single, force_accum, stream);
}

cake_status cake_rmsnorm_bwd_main(const cake_shape *shape, const cake_tensor *dy, const cake_tensor *x,
                                  const float *rstd, const void *w, cake_dtype w_dtype,
                                  const cake_tensor *dh, const cake_tensor *dx, float *dw,
                                  void *workspace, size_t workspace_bytes, int force_accum,
                                  cake_stream_t stream)
{
    return run_bwd(shape, dy, x, rstd, w, w_dtype, dh, dx, dw, workspace, workspace_bytes, 1, kFormPair,
                   force_accum, stream, kMainOnly);
}

cake_status cake_rmsnorm_bwd_reduce(const cake_shape *shape, int has_dh, float *dw, void *workspace,
                                    size_t workspace_bytes, cake_stream_t stream)
{
    uint32_t rows = 0;
    Plan plan;
    cake_status st = select_plan(shape, 1, has_dh, 0, -1, &plan, &rows);
    if (st != CAKE_OK)
        return st;
    if (!dw)
        return CAKE_ERR_INVALID;
    if (!aligned16(dw))
        return CAKE_ERR_UNSUPPORTED;
    const int H = (int)shape->hidden;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (rows == 0)
        return cuda_status(cudaMemsetAsync(dw, 0, (size_t)H * sizeof(float), s));
    if (!workspace || workspace_bytes < ws_size(H, plan.ctas, 1))
        return CAKE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return CAKE_ERR_UNSUPPORTED;
    const float2 *parts = reinterpret_cast<const float2 *>(static_cast<uint8_t *>(workspace) + ws_part_off(H));
    ReduceParams rp{parts, plan.ctas, H, dw, reduce_slices(H, plan.ctas)};
    return cuda_status(launch_dw_reduce(rp, s));
}

cake_status cake_rmsnorm_bwd_timeout_test(const cake_shape *shape, const cake_tensor *dy,
                                          const cake_tensor *x, const float *rstd, const void *w,
                                          cake_dtype w_dtype, const cake_tensor *dx, float *dw,
                                          void *workspace, size_t workspace_bytes,
                                          uint32_t wait_limit_us, cake_stream_t stream)
{
    if (wait_limit_us < 1 || wait_limit_us > 1000000)
        return CAKE_ERR_INVALID;
    // the grid barrier waits for CTA count + 1 arrivals: it never completes
    return run_bwd(shape, dy, x, rstd, w, w_dtype, nullptr, dx, dw, workspace, workspace_bytes, 1, kFormGrid, -1,
                   stream, kWhole, (uint64_t)wait_limit_us * 1000u, 1);
}

size_t cake_rmsnorm_bwd_host_staging_size(const cake_shape *shape, cake_dtype w_dtype, int has_dh, int chunks)
{
    uint32_t rows = 0;
    if (check_shape(shape, &rows) != CAKE_OK || rows == 0)
        return 0;
    HostChunking c;
    if (!host_chunking((int)shape->hidden, rows, has_dh != 0, w_dtype == CAKE_FP32 ? 4 : 2, chunks, &c))
        return 0;
    return c.total;
}

cake_status cake_rmsnorm_bwd_host(const cake_shape *shape, const void *dy, const void *x, const float *rstd,
                                  const void *w, cake_dtype w_dtype, const void *dh, void *dx, float *dw,
                                  void *staging, size_t staging_bytes, int chunks, int deterministic,
                                  cake_stream_t stream)
{
    (void)deterministic; // both modes run the pair: dw is reproducible either way
    return run_bwd_host(shape, dy, x, rstd, w, w_dtype, dh, dx, dw, staging, staging_bytes, chunks, stream);
}

cake_status cake_rmsnorm_plan_occupancy(const cake_shape *shape, int backward, int has_extra,
                                        int deterministic, int force_accum, int *planned,
                                        int *resident)
{
    if (!planned || !resident)
        return CAKE_ERR_INVALID;
    uint32_t rows = 0;
    Plan plan;
    cake_status st;
    if (backward) {
        st = select_plan(shape, deterministic, has_extra, -1, force_accum, &plan, &rows);
    } else {
        st = check_shape(shape, &rows);
        if (st == CAKE_OK)
            plan = make_plan((int)shape->hidden, rows, has_extra ? 2 : 1, kFwd, 0, 0);
    }
    if (st != CAKE_OK)
        return st;
    const int threads = 32 * (plan.groups * plan.rl.W + 1);
    int n = 0;
    cudaError_t e = backward ? occupancy_bwd(plan.rl.vpt, plan.rl.W, plan.rpg, plan.rl.lanes ? plan.rl.lanes : 32, plan.single, plan.dwm, threads, plan.smem, &n)
                             : occupancy_fwd(plan.rl.vpt, plan.rl.lanes ? plan.rl.lanes : 32, threads, plan.smem, &n);
    if (e != cudaSuccess)
        return CAKE_ERR_CUDA;
    *planned = plan.ctas_per_sm;
    *resident = n;
    return CAKE_OK;
}

cake_status cake_rmsnorm_device_status(int *code, int clear)
{
    if (!code)
        return CAKE_ERR_INVALID;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess)
        return CAKE_ERR_CUDA;
    int a = 0, b = 0;
    if (fwd_status(&a, clear) != cudaSuccess || bwd_status(&b, clear) != cudaSuccess)
        return CAKE_ERR_CUDA;
    *code = a ? a : b;
    return CAKE_OK;
}

} // extern "C"
