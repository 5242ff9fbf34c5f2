// Problem normalisation and launch planning (host only).
//
// Normalisation follows the host-argument record of "Composable Kernel:
// grouped_convolution_backward_weight_kernel.hpp Source File"
// (GroupedConvBwdWeightHostArgs: G_, N_, C_, K_, spatial lengths, strides,
// dilations, left/right pads).  That page takes the output lengths as an input;
// here they are derived with the standard rule and a caller-supplied value must
// agree with it.
//
// The implicit GEMM of that page (GemmM = K, GemmN = C*YX, GemmK = N*Ho*Wo,
// batched over G) is planned with the roles of M and N swapped for the tensor
// cores: MMA rows are (tap, channel) pairs -- the long axis -- and MMA columns
// are output channels k.
#include "plan.h"

#include <algorithm>
#include <array>
#include <vector>
#include <cmath>
#include <cstdio>
#include <cstdarg>
#include <cstring>

namespace wg {

namespace {

long long cdiv(long long a, long long b) { return (a + b - 1) / b; }
int round_up(int a, int b) { return (int)cdiv(a, b) * b; }
int pow2_at_least(int v)
{
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

int fail(std::string* err, int status, const char* fmt, ...) __attribute__((format(printf, 3, 4)));
int fail(std::string* err, int status, const char* fmt, ...)
{
    if (err) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        *err = buf;
    }
    return status;
}

// Candidate pixel tiles (w, h, d, n) for the tensor-core path: KT = product, a
// multiple of 16 (the MMA K of kind::f16) and at most 256; each extent at most
// the (rounded-up) extent of the pixel index space (Wo along w, or the wider
// shifted range of the x-taps-on-columns form).  With w8 the w extent is a
// multiple of 8, so that every 8-pixel K group is one contiguous run of a
// halo patch row.
void enumerate_tiles(const Problem& pb, int Wo, bool w8, std::vector<std::array<int, 4>>* out)
{
    const int Ho = pb.out[1], Do = pb.out[0], N = pb.N;
    const int lim_w = std::min(256 / pb.stride[2], round_up(Wo, w8 ? 8 : 16));
    const int lim_h = std::min(256 / pb.stride[1], pow2_at_least(Ho));
    const int lim_d = std::min(256 / pb.stride[0], pow2_at_least(Do));
    const int lim_n = std::min(256, pow2_at_least(N));
    out->clear();
    for (int bw = w8 ? 8 : 1; bw <= lim_w; bw += w8 ? 8 : 1)
        for (int bh = 1; bh <= lim_h && bw * bh <= 256; ++bh)
            for (int bd = 1; bd <= lim_d && bw * bh * bd <= 256; ++bd)
                for (int bn = 1; bn <= lim_n && bw * bh * bd * bn <= 256; ++bn)
                    if ((bw * bh * bd * bn) % 16 == 0) out->push_back({bw, bh, bd, bn});
}

// Stride phases of one spatial dim: tap t reads input offset t*dil = q*stride + ph.
struct DimPhases {
    int nph;
    int phval[8];
    int phidx[kMaxHaloFilter];
    int q[kMaxHaloFilter];
    int qmax;
};

bool dim_phases(int F, int s, int d, DimPhases* o)
{
    if (F > kMaxHaloFilter || s > 8) return false;
    bool used[8] = {false, false, false, false, false, false, false, false};
    o->qmax = 0;
    for (int t = 0; t < F; ++t) {
        used[(t * d) % s] = true;
        o->qmax = std::max(o->qmax, (t * d) / s);
    }
    o->nph = 0;
    int idx_of[8];
    for (int ph = 0; ph < s; ++ph)
        if (used[ph]) idx_of[ph] = o->nph, o->phval[o->nph++] = ph;
    for (int t = 0; t < F; ++t) o->phidx[t] = idx_of[(t * d) % s], o->q[t] = (t * d) / s;
    return true;
}

struct IgCand {
    int halo, box[4], nt[4], KT, mt, stages, stage_bytes, patch[3], patch_bytes, n_patches, dy_off;
    int xs, Nt, n_ntiles, n_katoms, n_atoms, n_mtiles, Nmma, dy_w, dy_bytes;
    int pair;
    long long tx_bytes;  // TMA bytes per K-tile and CTA
    long long cost, tile_clk, S;
};

// Cost terms of the split-K epilogue, in SM cycles (GB300 at ~2 GHz): L2
// takes ~2900 bytes per cycle device-wide; every kernel beyond the main one
// (the reduction of the two-stage path, the zeroing kernel of the atomic path)
// adds one launch, ~2.07 us per kernel in a stream of back-to-back calls
// (measured with empty kernels: 2.07 us per call for one kernel, 4.1 us for
// two); the cluster reduction writes the CTA's partial sums to shared memory
// and reads them back through distributed shared memory at ~12 B/cycle
// (measured), plus two cluster barriers.
constexpr long long kL2BytesPerClk = 2900;
constexpr long long kExtraLaunchClk = 4280;
// Cold reads from HBM, device-wide (~6 TB/s at ~2 GHz): no split degree reads
// the inputs faster than this.
constexpr long long kDramBytesPerClk = 3000;
// The CTA pair's extra cost per call (cluster launch, cluster barriers and the
// paired TMEM allocation and release), measured ~1 us.
constexpr long long kPairCallClk = 2100;

long long epilogue_clk(long long dw_bytes, int n_out, int Q, long long red_bytes, bool atomic)
{
    long long c = 0;
    if (Q > 1) c += red_bytes / 128 + red_bytes / 12 + 1500;
    if (atomic) {
        if (n_out > 1) c += (long long)n_out * dw_bytes / (kL2BytesPerClk / 3) + kExtraLaunchClk;
    } else if (n_out > 1) {
        c += 2 * (long long)n_out * dw_bytes / kL2BytesPerClk + kExtraLaunchClk;
    }
    return c;
}

int cap_index(int q) { return q == 1 ? 0 : q == 2 ? 1 : q == 4 ? 2 : 3; }

// Whether split partial sums are added with atomics: mode ATOMIC, or mode
// AUTO with an fp32 dW.  On GB300 the atomic path -- a zeroing kernel hidden
// behind the main loop, then one fp32 add per partial element -- measured
// faster than the two-stage one (partials written, a second kernel summing
// them) on every fp32 workload of the benchmark (the 56x56 workload with S =
// 75: 14.1 against 15.5 us).  A 16-bit dW takes the adds through an fp32 copy
// in the workspace and a third kernel that casts it, one more grid completion
// per call: 17.0 us there against 15.5 us two-stage, so AUTO keeps the
// two-stage path for it.  (Casting in the main kernel instead, by the last
// split CTA of each tile, put a 96 KB conversion by one CTA at the end of the
// call: 43.5 us.)
bool takes_atomic(const wg_options& o, const Problem& pb)
{
    return o.mode == WG_MODE_ATOMIC || (o.mode == WG_MODE_AUTO && pb.out_dtype == WG_FP32);
}

// Cycles the device needs to read the inputs once from HBM: all of dY, and the
// part of X that some tap reaches (along each dim a fraction of about
// min(1, dilated filter extent / stride) of the input positions: a quarter of
// X for a 1x1 filter with stride 2).
long long dram_read_clk(const Problem& pb)
{
    double frac = 1.0;
    for (int i = 0; i < 3; ++i) {
        const double extent = (double)(pb.filt[i] - 1) * pb.dil[i] + 1;
        frac *= std::min(1.0, extent / pb.stride[i]);
    }
    return (long long)(2.0 * ((double)pb.x_elems * frac + (double)pb.dy_elems) / kDramBytesPerClk);
}

// Split degree without clusters: the caller's, 1 for mode DIRECT, else enough
// splits of the K-tiles to fill the device once, evened out so that no split
// is short by more than one K-tile.
long long split_for(const wg_options& o, long long base, long long ktiles, const DeviceCaps& caps)
{
    if (o.split_k > 0) return o.split_k;
    if (o.mode == WG_MODE_DIRECT) return o.cluster > 1 ? o.cluster : 1;
    long long s = std::max(1LL, caps.cluster_ctas[0] / std::max(1LL, base));
    s = std::min(s, std::max(1LL, ktiles));
    const long long per = cdiv(ktiles, s);
    return cdiv(ktiles, per);
}

int plan_igemm(Plan* pl, const wg_options& o, const DeviceCaps& caps, std::string* err)
{
    const int num_sms = caps.num_sms;
    const Problem& pb = pl->pb;
    IgemmPlan& ig = pl->ig;
    std::memset(&ig, 0, sizeof ig);
    for (int j = 0; j < 3; ++j)
        if (pb.stride[j] > 8)
            return fail(err, WG_ERR_NOT_SUPPORTED, "stride above 8 (TMA element strides are at most 8)");
    // Channel / k windows.  A group whose first channel is not 8-aligned can
    // start up to 7 channels into the window (TMA coordinates must be 16-byte aligned).
    // The widest fold whose windows start 8-aligned (Gm*C and Gm*K multiples of
    // 8) is preferred; failing that, any width, with windows that may start up
    // to 7 channels early.
    int Gm = 1, cmis = (pb.C % 8) ? 7 : 0, kmis = (pb.K % 8) ? 7 : 0;
    for (int g = std::min(pb.G, 64); g >= 2; --g)
        if (g * pb.C <= 64 && g * pb.K <= 256 && (g * pb.C) % 8 == 0 && (g * pb.K) % 8 == 0) {
            Gm = g;
            cmis = kmis = 0;
            break;
        }
    if (Gm == 1 && pb.C + cmis <= 64 && pb.K + kmis <= 256)
        while (Gm < pb.G && (Gm + 1) * pb.C + cmis <= 64 && (Gm + 1) * pb.K + kmis <= 256) ++Gm;
    ig.Gm = Gm;
    ig.n_gblocks = (int)cdiv(pb.G, Gm);
    if (ig.n_gblocks > 65535) return fail(err, WG_ERR_NOT_SUPPORTED, "too many group blocks (%d)", ig.n_gblocks);
    ig.n_cchunks = (int)cdiv(Gm * pb.C + cmis, 64);
    const int kwin = Gm * pb.K + kmis;
    ig.n_ntiles = (int)cdiv(kwin, 256);
    ig.Nt = round_up((int)cdiv(kwin, ig.n_ntiles), 16);
    ig.n_katoms = (int)cdiv(ig.Nt, 64);
    if (pb.T * ig.n_cchunks > (1 << 24)) return fail(err, WG_ERR_NOT_SUPPORTED, "filter too large");
    ig.n_atoms = (int)(pb.T * ig.n_cchunks);
    ig.n_mtiles = (int)cdiv(ig.n_atoms, 2);

    // Stride phases per dim, in (w, h, d) order.
    DimPhases ph[3];
    bool ph_ok = true;
    for (int i = 0; i < 3; ++i) ph_ok = dim_phases(pb.filt[2 - i], pb.stride[2 - i], pb.dil[2 - i], &ph[i]) && ph_ok;
    bool halo_ok = ph_ok && ig.n_atoms <= kMaxHaloAtoms;
    const int n_combos = halo_ok ? ph[0].nph * ph[1].nph * ph[2].nph : 0;
    if (halo_ok && n_combos * ig.n_cchunks > kMaxPatches) halo_ok = false;

    // The x taps on the MMA columns (IgemmPlan::xs) need stride 1 (then a shift
    // of the pixel index along w is a shift of dY), whole 64-wide k atoms (a
    // folded tile keeps its block-diagonal mask in the epilogue), and at most
    // 256 columns.
    const int X = pb.filt[2], Y = pb.filt[1], Z = pb.filt[0];
    const char* mn_no = nullptr;
    if (pb.stride[0] != 1 || pb.stride[1] != 1 || pb.stride[2] != 1)
        mn_no = "stride 1 in every dim";
    else if (kwin % 64)
        mn_no = "a k window (K, or K times the groups folded into a tile) that is a multiple of 64";
    else if (X < 2 || X > 4)
        mn_no = "2 to 4 filter taps along w";
    else if (o.cluster > 1)
        mn_no = "no cluster reduction";
    else if (!ph_ok || ig.n_cchunks > kMaxPatches || (long long)Z * Y * ig.n_cchunks > kMaxHaloAtoms)
        mn_no = "one halo patch per channel chunk";
    if ((o.kernel == WG_KERNEL_IGEMM_TAPS_MN || o.kernel == WG_KERNEL_IGEMM_PAIR) && mn_no)
        return fail(err, WG_ERR_NOT_SUPPORTED, "the x-taps-on-columns tile needs %s", mn_no);
    // The CTA-pair form of it (igemm_wgrad_pair_kernel): a split's two M-tiles
    // (atoms y = 0, 1 and y = 2, 3 of one 64-channel chunk) on the two CTAs of
    // a cluster, rank r staging output channels 32r .. 32r+31 of dY.
    const char* pair_no = nullptr;
    if (mn_no)
        pair_no = mn_no;
    else if (Gm != 1 || kwin != 64)
        pair_no = "K = 64 without group folding";
    else if (ig.n_cchunks != 1)
        pair_no = "C <= 64";
    else if (Z != 1 || (Y != 3 && Y != 4))
        pair_no = "a 2-D filter with 3 or 4 taps along h";
    else if (caps.cluster_ctas[1] < 2)
        pair_no = "clusters of two CTAs at the kernel's shared-memory size";
    if (o.kernel == WG_KERNEL_IGEMM_PAIR && pair_no)
        return fail(err, WG_ERR_NOT_SUPPORTED, "the CTA-pair tile needs %s", pair_no);
    // Where the x taps can go on the columns and the k window is 64 wide, the
    // form with every tap on the rows (then N = 64) is taken only when asked
    // for: on the 56x56 C = K = 64 workload it measured slower at every split
    // degree (S = 1: 616 against 373 us; S = 4: 160 against 99 us; S = 75:
    // 25.3 against 21.1 us), although the cost model below rates it close at
    // low split degrees (its 128x64 MMAs and nine tap views per K-tile cost
    // more than the model charges).  Wider k windows give it N = 128-256
    // MMAs at the tensor rate, and the model chooses.
    const bool try_mn = !mn_no && o.kernel != WG_KERNEL_IGEMM_TAPS_M;
    const bool try_m = o.kernel == WG_KERNEL_IGEMM_TAPS_M ||
                       (!(try_mn && ig.Nt <= 64) && o.kernel != WG_KERNEL_IGEMM_TAPS_MN &&
                        o.kernel != WG_KERNEL_IGEMM_PAIR);
    const bool try_single_mn = o.kernel != WG_KERNEL_IGEMM_PAIR;
    const bool try_pair = !pair_no && o.kernel != WG_KERNEL_IGEMM_TAPS_MN && o.kernel != WG_KERNEL_IGEMM_TAPS_M;
    // Pairs resident at once (clusters must sit within one GPC).
    DeviceCaps caps_pair = caps;
    caps_pair.cluster_ctas[0] = caps.cluster_ctas[1] / 2 * 2;

    const int avail = kMaxSmemPerCta - 3072;
    IgCand best{};
    best.cost = -1;
    std::vector<std::array<int, 4>> tiles;
    // Forms: 2 = x taps on the columns (halo patches), 1 = every tap on the
    // rows with halo patches, 0 = every tap on the rows with per-tap boxes.
    for (int form = 2; form >= 0; --form) {
        if (form == 2 ? !try_mn : (!try_m || (form == 1 && !halo_ok))) continue;
        const bool mn = form == 2;
        const int halo = form >= 1 ? 1 : 0;
        IgCand f{};
        f.xs = mn ? X : 0;
        f.Nt = mn ? 64 : ig.Nt;
        f.n_ntiles = mn ? kwin / 64 : ig.n_ntiles;
        f.n_katoms = mn ? 1 : ig.n_katoms;
        f.n_atoms = mn ? Z * Y * ig.n_cchunks : ig.n_atoms;
        f.n_mtiles = (int)cdiv(f.n_atoms, 2);
        f.Nmma = mn ? 64 * X : ig.Nt;
        const int wq = mn ? pb.out[2] + (X - 1) * pb.dil[2] : pb.out[2];
        const int mt_max = std::min({f.n_mtiles, kMaxTmemCols / f.Nmma, kMaxMtPerCta});
        enumerate_tiles(pb, wq, halo != 0, &tiles);
        for (const auto& t : tiles) {
            IgCand c = f;
            c.halo = halo;
            for (int i = 0; i < 4; ++i) c.box[i] = t[i];
            c.nt[0] = (int)cdiv(wq, c.box[0]);
            c.nt[1] = (int)cdiv(pb.out[1], c.box[1]);
            c.nt[2] = (int)cdiv(pb.out[0], c.box[2]);
            c.nt[3] = (int)cdiv(pb.N, c.box[3]);
            c.KT = c.box[0] * c.box[1] * c.box[2] * c.box[3];
            const int slot = c.KT * 128;
            if (halo) {
                bool fits = true;
                for (int i = 0; i < 3; ++i) {
                    c.patch[i] = c.box[i] + (mn && i == 0 ? 0 : ph[i].qmax);
                    if (c.patch[i] * pb.stride[2 - i] > 256) fits = false;
                }
                if (!fits) continue;
                const long long rows = (long long)c.patch[0] * c.patch[1] * c.patch[2] * c.box[3];
                if (rows * 128 > avail) continue;
                c.patch_bytes = round_up((int)(rows * 128), 1024);
                c.n_patches = (mn ? 1 : n_combos) * ig.n_cchunks;
            } else {
                for (int i = 0; i < 3; ++i) c.patch[i] = c.box[i];
                c.patch_bytes = slot;
            }
            // dY staging: the K-tile's 64-channel boxes, or one patch widened
            // by the x taps' shifts.
            c.dy_w = mn ? c.box[0] + (X - 1) * pb.dil[2] : c.box[0];
            if (c.dy_w > 256) continue;
            const long long dy_bytes = mn ? (long long)c.dy_w * c.box[1] * c.box[2] * c.box[3] * 128
                                          : (long long)c.n_katoms * slot;
            if (dy_bytes > avail) continue;
            c.dy_bytes = (int)dy_bytes;
            const long long ktiles = (long long)c.nt[0] * c.nt[1] * c.nt[2] * c.nt[3];
            // mt M-tiles per CTA from mt_max down to 1, then (pr = 1) the CTA
            // pair: one M-tile per CTA, half of dY.
            for (int it = 0; it <= mt_max; ++it) {
                const int pr = it == mt_max ? 1 : 0;
                const int mt = pr ? 1 : mt_max - it;
                if (pr ? !(mn && try_pair) : (mn && !try_single_mn)) continue;
                const int n_x = halo ? c.n_patches : 2 * mt;
                // The pair's stage: [dY half][xshift][X patch]; xshift (atom 2's
                // row offset, 2 dil_h patch rows) must keep the X copies 1024-aligned.
                const long long dy_cta = pr ? c.dy_bytes / 2 : c.dy_bytes;
                const long long xshift = pr ? 2LL * pb.dil[1] * c.patch[0] * 128 : 0;
                if (xshift % 1024) continue;
                const long long stage = ((long long)n_x * c.patch_bytes + dy_cta + 1023) / 1024 * 1024 + xshift;
                // The single-CTA stage of the same tile (the pair is costed from it).
                const long long stage1 = ((long long)n_x * c.patch_bytes + c.dy_bytes + 1023) / 1024 * 1024;
                if (stage > avail || stage1 > avail) continue;
                const int stages = std::min(8, (int)(avail / stage));
                if (stages < 2) continue;
                // Stage bytes the TMA writes (the pair's gap is not written).
                const long long written = pr ? (long long)n_x * c.patch_bytes + dy_cta : stage;
                // Per K-tile and CTA: the MMAs -- each the longer of the tensor
                // pipe (N/2 cycles) and its shared-memory reads (A 4 KB + B 32*N
                // bytes at ~128 B/cycle) -- against the stage's fill at ~40
                // B/cycle (every SM loading at once; calibrated on the 56x56
                // workload, where 2, 3 and 5 M-tiles per CTA measured 27.6,
                // 24.7 and 26.5 us), plus a fixed overhead; fewer than 3 stages
                // exposes latency.
                // With the x taps on the columns the MMAs' operand reads and
                // the stage's TMA writes share the SM's shared-memory
                // bandwidth, so a tile with less halo (fewer stage bytes per
                // pixel) costs less although the tensor pipe would tie (grouped
                // G = 32: a 32 x 4 pixel tile 14.7 us against 14.9-15.1 us for
                // 8 x 2 x 8 images; 8 x 14 measured 14.4 us).  Charging the
                // stage bytes to the plans with every tap on the rows as well
                // moved three 5x5 depthwise folds to tiles that ran 3-12%
                // slower, so there the MMA term stays alone.
                const long long mranges = cdiv(c.n_mtiles, mt);
                const long long ksteps = c.KT / 16;
                const long long mma_one = std::max<long long>(c.Nmma / 2, 32 + c.Nmma / 4);
                const long long smem_clk = (long long)mt * ksteps * (32 + c.Nmma / 4) + stage1 / 128;
                const long long mma_clk = std::max((long long)mt * ksteps * mma_one, mn ? smem_clk : 0LL);
                const long long load_clk = stage1 / 40;
                long long tile_clk = std::max(mma_clk, load_clk) + 64;
                // Fewer than 3 stages exposes the refill latency -- when the
                // split has more K-tiles than the ring holds (below).
                const bool few_stages = (pr ? stages : std::min(8, (int)(avail / stage1))) < 3;
                // The CTA pair halves each SM's operand reads of B and its dY
                // loads, but on the 56x56 workload its K-tile measured only
                // 3.5% shorter than the single CTA's (0.804 against 0.833 us
                // with one split; equal with 75 splits, when the memory system
                // rather than the SM bounds the loop), and its cluster launch,
                // barriers and paired TMEM release cost ~1 us per call
                // (kPairCallClk, added to the call's cost below): it pays for
                // long splits only (S = 1 and 4: 360 and 97 us against 373 and
                // 99; S = 38 and 75: 20.1 and 16.2 us against 19.1 and 15.5).
                if (pr) tile_clk = tile_clk * 965 / 1000;
                // Whole-call estimate for the split degrees this tiling may get
                // (the caller's; else enough splits to fill the device once, or
                // 3/4, 2/3 or 1/2 of that): the K-tiles of one split in waves of
                // resident CTAs -- but no faster than the device reads the inputs
                // from HBM -- plus the partial sums that the splits write and the
                // reduction reads back.  Fewer splits pay when the cold read, not
                // the per-SM loads, bounds the main loop (1x1 C 64 -> K 256:
                // 23.3-23.8 us with S = 75-100 against 24.8 us with S = 150).
                const long long base = mranges * c.n_ntiles * ig.n_gblocks;
                const DeviceCaps& cp = pr ? caps_pair : caps;
                const long long s_fill = split_for(o, base, ktiles, cp);
                const bool auto_s = o.split_k == 0 && o.mode != WG_MODE_DIRECT && o.cluster <= 1;
                const bool atomic_sum = takes_atomic(o, pb);
                const long long dram_clk = dram_read_clk(pb);
                const long long red_bytes = (long long)mt * c.Nmma * 512;
                for (int fi = 0; fi < (auto_s ? 4 : 1); ++fi) {
                    static const int num[4] = {1, 3, 2, 1}, den[4] = {1, 4, 3, 2};
                    long long S = std::max(1LL, s_fill * num[fi] / den[fi]);
                    if (fi > 0) S = cdiv(ktiles, cdiv(ktiles, S));  // splits of whole, even K-tile counts
                    // The per-CTA estimate also breaks ties between tilings whose
                    // main loops all sit under the HBM bound (with weight 1/8).
                    const long long waves = cdiv(base * S, cp.cluster_ctas[0]);
                    // A split whose K-tiles all fit the ring issues every load at
                    // once: no refill waits (3-D stride 2, S = 8: two 128-pixel
                    // K-tiles in two stages, 11.9 us atomic and 15.0 us two-stage,
                    // against four 64-pixel K-tiles of six 8 KB boxes, ~1.5 us
                    // each, that the penalty used to pick: 14.5 and 17.7 us).
                    const long long kper = cdiv(ktiles, S);
                    const long long tclk = few_stages && kper > stages ? tile_clk * 13 / 10 : tile_clk;
                    const long long main_clk = waves * kper * tclk;
                    const long long cost = std::max(main_clk, dram_clk) + main_clk / 8 + (pr ? kPairCallClk : 0) +
                                           epilogue_clk(pb.dw_elems * 4, (int)S, 1, red_bytes, atomic_sum);
                    // With the x taps on the columns, ties go to the fewer TMA
                    // bytes per K-tile (fewer bytes through L2; among the tilings
                    // of the other form this moved 5x5 depthwise folds to slower
                    // tiles, as the shared-memory charge above did).
                    // Ties within one wave of CTAs go to fewer M-tiles per CTA:
                    // more CTAs, each with a shorter epilogue (8x8 C 16 -> K 32,
                    // one K-tile: 2 CTAs of 3 M-tiles 18.5 us against 16.4 us
                    // for 5 CTAs of 1).
                    const bool fewer_mt = waves == 1 && mt < best.mt;
                    if (best.cost < 0 || cost < best.cost ||
                        (cost == best.cost && (fewer_mt || (mn && best.xs && mt == best.mt && written < best.tx_bytes)))) {
                        c.mt = mt;
                        c.stages = stages;
                        c.stage_bytes = (int)stage;
                        c.dy_off = n_x * c.patch_bytes;
                        c.pair = pr;
                        c.tx_bytes = written;
                        c.cost = cost;
                        c.tile_clk = tclk;
                        c.S = S;
                        best = c;
                    }
                }
            }
        }
    }
    if (best.cost < 0) return fail(err, WG_ERR_NOT_SUPPORTED, "no tile configuration fits shared memory");
    ig.halo = best.halo;
    ig.xs = best.xs;
    ig.Nt = best.Nt;
    ig.n_ntiles = best.n_ntiles;
    ig.n_katoms = best.n_katoms;
    ig.n_atoms = best.n_atoms;
    ig.n_mtiles = best.n_mtiles;
    ig.Nmma = best.Nmma;
    ig.dy_w = best.dy_w;
    ig.pair = best.pair;
    // A CTA of the pair stages 32 of the 64 output channels of the dY patch.
    ig.dy_bytes = ig.pair ? best.dy_bytes / 2 : best.dy_bytes;
    std::memcpy(ig.box, best.box, sizeof best.box);
    std::memcpy(ig.ntile, best.nt, sizeof best.nt);
    std::memcpy(ig.patch, best.patch, sizeof best.patch);
    ig.KT = best.KT;
    ig.slot_bytes = best.KT * 128;
    ig.patch_bytes = best.patch_bytes;
    ig.n_mranges = (int)cdiv(ig.n_mtiles, best.mt);
    ig.mt_per_cta = (int)cdiv(ig.n_mtiles, ig.n_mranges);
    ig.n_patches = ig.halo ? best.n_patches : 2 * ig.mt_per_cta;
    ig.dy_off = ig.n_patches * ig.patch_bytes;
    ig.stage_bytes = round_up(ig.dy_off + ig.dy_bytes, 1024);
    if (ig.pair) {
        // [dY half][xshift][X patch] (rank 1's X copy xshift bytes lower).
        ig.pair_xshift = 2 * pb.dil[1] * ig.patch[0] * 128;
        ig.dy_off = 0;
        ig.pair_xoff = round_up(ig.dy_bytes, 1024) + ig.pair_xshift;
        ig.stage_bytes = ig.pair_xoff + ig.patch_bytes;
    }
    ig.stages = std::min(8, avail / ig.stage_bytes);
    // Stage buffers, then 1 KB of slack that a padding atom's reads may reach,
    // then 1 KB of barriers and tables; plus 1 KB to align the base.
    ig.smem_bytes = ig.stages * ig.stage_bytes + 3072;
    ig.tmem_cols = std::max(32, pow2_at_least(ig.mt_per_cta * ig.Nmma));
    ig.total_kt = (long long)ig.ntile[0] * ig.ntile[1] * ig.ntile[2] * ig.ntile[3];
    ig.est_cycles = best.cost / std::max(1, num_sms);
    ig.tile_clk = best.tile_clk;
    if (ig.total_kt > (1ll << 31) - 1) return fail(err, WG_ERR_NOT_SUPPORTED, "GemmK too large");
    if (ig.halo) {
        for (int i = 0; i < 3; ++i) ig.n_phase[i] = ph[i].nph;
        // Patches in (phase d, phase h, phase w, chunk) order; atoms sorted by
        // their offset in the stage so that the two atoms of an M-tile are a
        // non-negative LBO apart.
        int p = 0;
        for (int a = 0; a < ph[2].nph; ++a)
            for (int b = 0; b < ph[1].nph; ++b)
                for (int cph = 0; cph < ph[0].nph; ++cph)
                    for (int cc = 0; cc < ig.n_cchunks; ++cc, ++p) {
                        ig.patch_ph[p][0] = (unsigned char)ph[0].phval[cph];
                        ig.patch_ph[p][1] = (unsigned char)ph[1].phval[b];
                        ig.patch_ph[p][2] = (unsigned char)ph[2].phval[a];
                        ig.patch_ph[p][3] = (unsigned char)cc;
                    }
        struct At { unsigned off; int tap, cc; };
        At at[kMaxHaloAtoms];
        int na = 0;
        // With the x taps on the columns an atom is (z, y, chunk) and its tap
        // entry is that of x = 0; the epilogue adds each column block's x.
        const int XA = ig.xs ? 1 : X;
        for (int z = 0; z < Z; ++z)
            for (int y = 0; y < Y; ++y)
                for (int x = 0; x < XA; ++x)
                    for (int cc = 0; cc < ig.n_cchunks; ++cc) {
                        const int combo = (ph[2].phidx[z] * ph[1].nph + ph[1].phidx[y]) * ph[0].nph + ph[0].phidx[x];
                        const int patch = combo * ig.n_cchunks + cc;
                        const long long qoff =
                            ((long long)ph[2].q[z] * ig.patch[1] + ph[1].q[y]) * ig.patch[0] + ph[0].q[x];
                        at[na].off = (unsigned)(patch * ig.patch_bytes + qoff * 128);
                        at[na].tap = (z * Y + y) * X + x;
                        at[na].cc = cc;
                        ++na;
                    }
        std::stable_sort(at, at + na, [](const At& l, const At& r) { return l.off < r.off; });
        for (int i = 0; i < na; ++i) {
            ig.atom_off[i] = at[i].off;
            ig.atom_tap[i] = (unsigned short)at[i].tap;
            ig.atom_cc[i] = (unsigned char)at[i].cc;
        }
        if (ig.pair) {
            // Rank 1's X copy sits pair_xshift bytes lower, so that its atoms
            // (y = 2, 3) are read at the offsets of rank 0's (y = 0, 1): the
            // pair shares one A descriptor.  Atoms y are dil_h rows apart.
            const unsigned d1 = ig.atom_off[1] - ig.atom_off[0], d2 = ig.atom_off[2] - ig.atom_off[0];
            if (na < 3 || ig.atom_off[0] != 0 || d2 != (unsigned)ig.pair_xshift || d2 != 2 * d1 ||
                (na == 4 && ig.atom_off[3] - ig.atom_off[0] != 3 * d1))
                return fail(err, WG_ERR_NOT_SUPPORTED, "CTA-pair atoms are not evenly spaced");
        }
    }

    const long long base = (long long)ig.n_mranges * ig.n_ntiles * ig.n_gblocks;
    if (base > 65535LL * 65535LL) return fail(err, WG_ERR_NOT_SUPPORTED, "grid too large");
    // Cluster reduction: the CTA's partial sums (mt_per_cta * Nt columns of 128
    // fp32 rows) are staged in its pipeline buffers.
    const long long red_bytes = (long long)ig.mt_per_cta * ig.Nmma * 128 * 4;
    const bool cl_ok = red_bytes <= (long long)ig.stages * ig.stage_bytes;
    if (o.cluster > 1 && !cl_ok)
        return fail(err, WG_ERR_NOT_SUPPORTED,
                    "cluster reduction: the CTA's partial sums (%lld bytes) do not fit its shared memory", red_bytes);
    const long long dw_bytes = pb.dw_elems * 4;
    const bool atomic = takes_atomic(o, pb);
    int S, Q;
    if (o.split_k > 0) {
        S = o.split_k;
        Q = o.cluster > 0 ? o.cluster : 1;
        if (S % Q) return fail(err, WG_ERR_INVALID_ARGUMENT, "cluster %d does not divide split_k %d", Q, S);
    } else if (o.mode == WG_MODE_DIRECT) {
        S = Q = o.cluster > 1 ? o.cluster : 1;
    } else {
        // Fill the device in one wave for each cluster size, then keep the
        // cheapest by the planner's cycle estimate.  Automatic plans use no
        // clusters: distributed shared memory moves ~10-14 bytes per cycle per
        // SM on GB300 (measured), so the cluster reduction was slower than
        // writing the partial sums to L2 on every workload measured.
        S = Q = 0;
        long long best_clk = -1;
        for (int q = 1; q <= 8; q *= 2) {
            if (o.cluster > 0 ? q != o.cluster : q != 1) continue;
            if (q > 1 && !cl_ok) continue;
            const long long fit = caps.cluster_ctas[cap_index(q)] / (base * q);
            long long s = q == 1 && o.cluster <= 1 ? best.S : q * std::max(1LL, fit);
            s = std::min<long long>(s, round_up((int)std::min<long long>(ig.total_kt, 1 << 20), q));
            const long long per = cdiv(ig.total_kt, s);
            s = std::min<long long>(65535 / q * q, round_up((int)cdiv(ig.total_kt, per), q));
            const long long clk = cdiv(ig.total_kt, s) * ig.tile_clk +
                                  epilogue_clk(dw_bytes, (int)(s / q), q, red_bytes, atomic);
            if (best_clk < 0 || clk < best_clk) best_clk = clk, S = (int)s, Q = q;
        }
    }
    if (S > 65535) return fail(err, WG_ERR_NOT_SUPPORTED, "split_k %d above 65535", S);
    ig.cluster = Q;
    pl->S = S;
    pl->per_split = cdiv(ig.total_kt, S);
    pl->grid[0] = (unsigned)(ig.n_mranges * ig.n_ntiles);
    pl->grid[1] = (unsigned)ig.n_gblocks;
    pl->grid[2] = (unsigned)S;
    pl->block = 256;  // the kernel's thread count (kIgThreads)
    return WG_OK;
}

bool dw_eligible(const Problem& pb)
{
    if (pb.C != 1 || pb.K != 1 || pb.ndim > 2 || pb.T > 9 || pb.G % 8) return false;
    const int wspan = (pb.out[2] - 1) * pb.stride[2] + (pb.filt[2] - 1) * pb.dil[2] + 1;
    return wspan <= 256 && pb.out[2] <= 256;
}

int plan_depthwise(Plan* pl, const wg_options& o, int num_sms, std::string* err)
{
    if (o.cluster > 1)
        return fail(err, WG_ERR_NOT_SUPPORTED, "cluster > 1 is for the tensor-core kernel (the depthwise kernel has none)");
    const Problem& pb = pl->pb;
    DwPlan& dw = pl->dw;
    std::memset(&dw, 0, sizeof dw);
    // Channel vector of Gm channels (the caller's merge degree; make_plan picks
    // the automatic one).
    dw.Gm = o.group_merge > 0 ? o.group_merge : 2;
    const int Wo = pb.out[2], Ho = pb.out[1];
    dw.xw = (Wo - 1) * pb.stride[2] + (pb.filt[2] - 1) * pb.dil[2] + 1;
    // Two CTAs per SM when the channel vector is at most 4 wide (register use
    // allows it): half the shared memory each.
    const int ctas_per_sm = dw.Gm <= 4 ? 2 : 1;
    const int avail = (ctas_per_sm == 2 ? kMaxSmemPerCta / 2 - 2048 : kMaxSmemPerCta) - 1024 - 512;
    // Channels per CTA (64, 32 or 16) and rows per tile: the fewest X and dY
    // elements loaded per channel over the image (X rows are re-read across a
    // tile's halo, and padded rows are wasted), with at least 3 stages and at
    // most 256 compute threads; ties go to more channels, then taller tiles.
    int bestR = 0, bestCB = 0, prevCB = 0;
    long long best = -1;
    for (int cb = 64; cb >= 16; cb /= 2) {
        const int CB = std::min(cb, round_up(pb.G, 8));
        if (CB == prevCB || CB < dw.Gm || CB % dw.Gm) continue;
        prevCB = CB;
        const int NV = CB / dw.Gm;
        for (int R = std::min(8, Ho); R >= 1; --R) {
            if (NV * R > 256) continue;
            const int xh = (R - 1) * pb.stride[1] + (pb.filt[1] - 1) * pb.dil[1] + 1;
            if (xh > 256) continue;
            const int stage = CB * 2 * (dw.xw * xh + Wo * R);
            if (avail / stage < 3) continue;
            const long long loads = cdiv(Ho, R) * ((long long)xh * dw.xw + (long long)R * Wo);
            const long long cost = loads * 1000 + (64 - CB) * 10 + (8 - R);
            if (best < 0 || cost < best) best = cost, bestR = R, bestCB = CB;
        }
    }
    if (!bestR) return fail(err, WG_ERR_NOT_SUPPORTED, "depthwise tile does not fit shared memory");
    dw.CB = bestCB;
    dw.n_cblocks = (int)cdiv(pb.G, dw.CB);
    const int NV = dw.CB / dw.Gm;
    dw.R = bestR;
    dw.xh = (dw.R - 1) * pb.stride[1] + (pb.filt[1] - 1) * pb.dil[1] + 1;
    dw.nseg = std::max(1, std::min(Wo, 256 / (NV * dw.R)));
    dw.seg_len = (int)cdiv(Wo, dw.nseg);
    dw.nseg = (int)cdiv(Wo, dw.seg_len);
    dw.threads = round_up(NV * dw.R * dw.nseg, 32);
    dw.x_bytes = dw.CB * 2 * dw.xw * dw.xh;
    dw.dy_bytes = dw.CB * 2 * Wo * dw.R;
    dw.stage_bytes = round_up(dw.x_bytes, 128) + round_up(dw.dy_bytes, 128);
    dw.stages = std::min(ctas_per_sm == 2 ? 4 : 6, avail / dw.stage_bytes);
    const int red_bytes = dw.threads * (int)pb.T * dw.Gm * 4;
    dw.smem_bytes = std::max(dw.stages * dw.stage_bytes, red_bytes) + 1024 + 512;
    if (dw.smem_bytes > kMaxSmemPerCta) return fail(err, WG_ERR_NOT_SUPPORTED, "depthwise reduction too large");
    dw.sliding = (pb.stride[2] == 1 && pb.dil[2] == 1) ? 1 : 0;
    dw.total_tiles = (long long)pb.N * cdiv(Ho, dw.R);
    int S;
    if (o.split_k > 0) {
        S = o.split_k;
    } else if (o.mode == WG_MODE_DIRECT) {
        S = 1;
    } else {
        S = (int)std::max(1LL, (long long)std::llround((double)num_sms * ctas_per_sm / (double)dw.n_cblocks));
        S = (int)std::min<long long>(S, dw.total_tiles);
        S = std::min(S, 65535);
        const long long per = cdiv(dw.total_tiles, S);
        S = (int)cdiv(dw.total_tiles, per);
    }
    if (S > 65535) return fail(err, WG_ERR_NOT_SUPPORTED, "split_k %d above 65535", S);
    pl->S = S;
    pl->per_split = cdiv(dw.total_tiles, S);
    pl->grid[0] = (unsigned)dw.n_cblocks;
    pl->grid[1] = (unsigned)S;
    pl->grid[2] = 1;
    pl->block = (unsigned)(dw.threads + 32);
    return WG_OK;
}

}  // namespace

int normalize(const wg_problem* p, Problem* o, std::string* err)
{
    if (!p) return fail(err, WG_ERR_INVALID_ARGUMENT, "problem is NULL");
    std::memset(o, 0, sizeof *o);
    if (p->ndim < 1 || p->ndim > 3) return fail(err, WG_ERR_INVALID_ARGUMENT, "ndim must be 1, 2 or 3 (got %d)", p->ndim);
    if (p->G < 1 || p->N < 1 || p->C < 1 || p->K < 1)
        return fail(err, WG_ERR_INVALID_ARGUMENT, "G, N, C, K must be positive");
    if (p->in_dtype != WG_BF16 && p->in_dtype != WG_FP16)
        return fail(err, WG_ERR_INVALID_ARGUMENT, "in_dtype must be WG_BF16 or WG_FP16");
    if (p->out_dtype != WG_FP32 && p->out_dtype != WG_BF16 && p->out_dtype != WG_FP16)
        return fail(err, WG_ERR_INVALID_ARGUMENT, "out_dtype must be WG_FP32, WG_BF16 or WG_FP16");
    o->ndim = p->ndim;
    o->G = p->G, o->N = p->N, o->C = p->C, o->K = p->K;
    o->in_dtype = p->in_dtype, o->out_dtype = p->out_dtype;
    const int off = 3 - p->ndim;
    for (int i = 0; i < 3; ++i) {
        o->in[i] = o->filt[i] = o->out[i] = o->stride[i] = o->dil[i] = 1;
        o->pad_l[i] = o->pad_r[i] = 0;
    }
    for (int i = 0; i < p->ndim; ++i) {
        const int j = off + i;
        if (p->in[i] < 1 || p->filt[i] < 1 || p->stride[i] < 1 || p->dil[i] < 1 || p->pad_l[i] < 0 || p->pad_r[i] < 0)
            return fail(err, WG_ERR_INVALID_ARGUMENT,
                        "spatial dim %d: in, filt, stride, dil must be >= 1 and pads >= 0", i);
        const long long num = (long long)p->in[i] + p->pad_l[i] + p->pad_r[i] - (long long)p->dil[i] * (p->filt[i] - 1) - 1;
        if (num < 0)
            return fail(err, WG_ERR_INVALID_ARGUMENT, "spatial dim %d: dilated filter larger than padded input", i);
        const long long out = num / p->stride[i] + 1;
        if (out > (1 << 30)) return fail(err, WG_ERR_INVALID_ARGUMENT, "spatial dim %d: output too large", i);
        if (p->out[i] != 0 && p->out[i] != out)
            return fail(err, WG_ERR_INVALID_ARGUMENT, "spatial dim %d: out=%d but the derived length is %lld", i,
                        p->out[i], out);
        o->in[j] = p->in[i], o->filt[j] = p->filt[i], o->out[j] = (int)out;
        o->stride[j] = p->stride[i], o->dil[j] = p->dil[i], o->pad_l[j] = p->pad_l[i], o->pad_r[j] = p->pad_r[i];
    }
    o->T = (long long)o->filt[0] * o->filt[1] * o->filt[2];
    o->P = (long long)o->N * o->out[0] * o->out[1] * o->out[2];
    o->x_elems = (long long)o->N * o->in[0] * o->in[1] * o->in[2] * o->G * o->C;
    o->dy_elems = o->P * o->G * o->K;
    o->dw_elems = (long long)o->G * o->K * o->T * o->C;
    const long long lim = (1ll << 31) - 1;
    if (o->x_elems > lim || o->dy_elems > lim || o->dw_elems > lim)
        return fail(err, WG_ERR_NOT_SUPPORTED, "a tensor has 2^31 or more elements");
    return WG_OK;
}

DeviceCaps default_caps(int num_sms)
{
    if (num_sms <= 0) num_sms = kDefaultSMs;
    DeviceCaps c;
    c.num_sms = num_sms;
    c.cluster_ctas[0] = num_sms;
    c.cluster_ctas[1] = num_sms;
    c.cluster_ctas[2] = num_sms * 144 / 152;
    c.cluster_ctas[3] = num_sms * 120 / 152;
    return c;
}

int make_plan(const wg_problem* p, const wg_options* opt, const DeviceCaps& caps_in, Plan* pl, std::string* err)
{
    std::memset(pl, 0, sizeof *pl);
    int st = normalize(p, &pl->pb, err);
    if (st) return st;
    const Problem& pb = pl->pb;
    wg_options o{0, WG_MODE_AUTO, 0, 0, WG_KERNEL_AUTO};
    if (opt) o = *opt;
    DeviceCaps caps = caps_in;
    if (caps.num_sms <= 0) caps = default_caps(0);
    for (int i = 0; i < 4; ++i)
        if (caps.cluster_ctas[i] <= 0) caps.cluster_ctas[i] = default_caps(caps.num_sms).cluster_ctas[i];
    const int num_sms = caps.num_sms;
    if (o.split_k < 0) return fail(err, WG_ERR_INVALID_ARGUMENT, "split_k must be >= 0");
    if (o.mode < WG_MODE_AUTO || o.mode > WG_MODE_DETERMINISTIC) return fail(err, WG_ERR_INVALID_ARGUMENT, "bad mode");
    if (o.group_merge != 0 && o.group_merge != 1 && o.group_merge != 2 && o.group_merge != 4 && o.group_merge != 8)
        return fail(err, WG_ERR_INVALID_ARGUMENT, "group_merge must be 0, 1, 2, 4 or 8");
    if (o.cluster != 0 && o.cluster != 1 && o.cluster != 2 && o.cluster != 4 && o.cluster != 8)
        return fail(err, WG_ERR_INVALID_ARGUMENT, "cluster must be 0, 1, 2, 4 or 8");
    if (o.kernel < WG_KERNEL_AUTO || o.kernel > WG_KERNEL_IGEMM_PAIR)
        return fail(err, WG_ERR_INVALID_ARGUMENT, "bad kernel selector");
    if (o.mode == WG_MODE_DIRECT && o.split_k > 1 && o.split_k != o.cluster)
        return fail(err, WG_ERR_INVALID_ARGUMENT,
                    "mode DIRECT takes no split, or exactly one cluster of splits (split_k %d, cluster %d)", o.split_k,
                    o.cluster);
    if (((long long)pb.G * pb.C * 2) % 16 || ((long long)pb.G * pb.K * 2) % 16)
        return fail(err, WG_ERR_NOT_SUPPORTED, "G*C and G*K must be multiples of 8 (16-byte pixel rows for TMA)");
    const bool depthwise = pb.C == 1 && pb.K == 1;
    if (o.group_merge > 1 && !depthwise)
        return fail(err, WG_ERR_NOT_SUPPORTED, "group_merge > 1 is for depthwise problems (C = K = 1) only");
    const bool use_dw =
        depthwise && dw_eligible(pb) && (o.kernel == WG_KERNEL_AUTO || o.kernel == WG_KERNEL_DEPTHWISE);
    if (o.kernel == WG_KERNEL_DEPTHWISE && !use_dw)
        return fail(err, WG_ERR_NOT_SUPPORTED,
                    "the depthwise kernel needs C = K = 1, 1-D or 2-D, <= 9 taps and G %% 8 == 0");
    if (use_dw) {
        pl->kind = KIND_DEPTHWISE;
        // Automatic merge degree.  The PR #12359 page's policy (PR #12951)
        // takes the largest admissible Gm at the kernel's tile; here the
        // vector is two channels, one packed 32-bit word: every load moves a
        // pair and every mixed-precision multiply-add pair reads one word.
        // Wider vectors cut the load instructions per multiply-add further,
        // but with the per-tile work of the loop reduced to its loads and
        // multiply-adds the main loop runs at the DRAM rate either way, while
        // a wider vector lengthens the end of every CTA (9*Gm accumulators per
        // thread through the shuffle reduction) and shortens the column
        // segments (more segment starts and ragged tails).  Measured with the
        // policy sweep over 16 shapes (bench.py --sweep): two channels best or
        // within a few percent on the 3x3 shapes.  One channel when a
        // two-channel tile does not fit.
        if (o.group_merge == 0) {
            st = WG_ERR_NOT_SUPPORTED;
            for (int g = 2; g >= 1 && st != WG_OK; g /= 2) {
                wg_options og = o;
                og.group_merge = g;
                st = plan_depthwise(pl, og, num_sms, g == 1 ? err : nullptr);
            }
        } else {
            st = plan_depthwise(pl, o, num_sms, err);
        }
    } else {
        if (o.group_merge > 1)
            return fail(err, WG_ERR_NOT_SUPPORTED,
                        "group_merge > 1 needs the depthwise kernel (1-D/2-D, <= 9 taps, G %% 8 == 0)");
        pl->kind = KIND_IGEMM;
        st = plan_igemm(pl, o, caps, err);
    }
    if (st) return st;
    // Partial sums that reach memory per dW element: one per cluster of splits.
    const int n_out = pl->kind == KIND_IGEMM ? pl->S / pl->ig.cluster : pl->S;
    if (o.mode == WG_MODE_ATOMIC)
        pl->mode = MODE_ATOMIC;
    else if (n_out == 1)
        pl->mode = MODE_DIRECT;
    else if (takes_atomic(o, pb))
        pl->mode = MODE_ATOMIC;
    else
        pl->mode = MODE_DETERMINISTIC;
    // Workspace rows: one per (g, k) of T*C elements for the tensor-core kernel
    // (its epilogue walks dW rows), the whole of dW as one row for the
    // depthwise kernel.  Slices of at most 128 elements, a multiple of 4: the
    // whole row when it is that short, else the widest such width from 64 to
    // 128 that divides the row (no padding), else 128.
    pl->n_out = n_out;
    if (pl->kind == KIND_IGEMM) {
        // Staged output for folded groups: the CTA covers whole groups -- one
        // M-range, one N-tile, channel and k windows starting at the first
        // channel of their first group -- so its results are one contiguous
        // block of dW, Gm*K*T*C elements, of which the block-diagonal mask
        // keeps one element in Gm of the tile.  The accumulators are dumped
        // into the idle pipeline buffers and the block is written in dW order
        // four channels at a time (C a multiple of 4, so a vector never leaves
        // its 64-channel atom or, in the workspace, its slice of a dW row).
        // Measured on the grouped G = 32, C = K = 8 workload: 19.8 -> 16.5 us
        // (atomic), 20.5 -> 19.9 us (two-stage); for an unfolded tile (the 1x1
        // C 64 -> K 256 workload, every element kept) the per-element
        // epilogue was faster (20.5 against 22.6 us), so unfolded tiles keep it.
        // Split modes only: a single split of whole groups (direct mode) keeps
        // the per-element epilogue.
        const IgemmPlan& ig = pl->ig;
        const long long dump = (long long)ig.mt_per_cta * ig.Nmma * 128 * 4;
        const bool whole = ig.n_mranges == 1 && ig.n_ntiles == 1 && ig.cluster == 1 && (ig.Gm * pb.C) % 8 == 0 &&
                           (ig.Gm * pb.K) % 8 == 0;
        pl->ig.staged = ig.Gm > 1 && pl->mode != MODE_DIRECT && whole && pb.C % 4 == 0 &&
                                dump <= (long long)ig.stages * ig.stage_bytes
                            ? 1
                            : 0;
        // The kernel instance compiled for the most common stride-1 family (see
        // igemm_wgrad_kernel): x taps on the columns, one M-tile per CTA, a
        // split mode.
        pl->ig.spec = ig.pair ? 2 : ig.xs > 0 && ig.mt_per_cta == 1 && pl->mode != MODE_DIRECT ? 1 : 0;
    }
    pl->ws_rows = pl->kind == KIND_IGEMM ? (long long)pb.G * pb.K : 1;
    pl->ws_L = pb.dw_elems / pl->ws_rows;
    if (pl->ws_L <= 128) {
        pl->ws_W = round_up((int)pl->ws_L, 4);
    } else {
        pl->ws_W = 128;
        for (int w = 128; w >= 64; w -= 4)
            if (pl->ws_L % w == 0) {
                pl->ws_W = w;
                break;
            }
    }
    pl->ws_nj = (int)cdiv(pl->ws_L, pl->ws_W);
    pl->ws_bytes = pl->mode == MODE_DETERMINISTIC
                       ? (size_t)pl->ws_rows * pl->ws_nj * (size_t)n_out * pl->ws_W * 4
                       : 0;
    // Atomic accumulation of a 16-bit dW: an fp32 copy of dW in the workspace.
    pl->acc_ws = pl->mode == MODE_ATOMIC && pb.out_dtype != WG_FP32 ? 1 : 0;
    if (pl->acc_ws) pl->ws_bytes = (size_t)((pb.dw_elems + 3) / 4) * 16;
    return WG_OK;
}

std::string plan_string(const Plan& pl)
{
    const Problem& pb = pl.pb;
    char buf[1024];
    const char* mode = pl.mode == MODE_DIRECT ? "direct" : pl.mode == MODE_ATOMIC ? "atomic" : "deterministic";
    if (pl.kind == KIND_IGEMM) {
        const IgemmPlan& ig = pl.ig;
        snprintf(buf, sizeof buf,
                 "kernel=igemm_tcgen05 %s taps=%s Nmma=%d mode=%s S=%d cluster=%d Gm=%d gblocks=%d cchunks=%d "
                 "Nt=%d ntiles=%d "
                 "katoms=%d "
                 "box=(w%d,h%d,d%d,n%d) KT=%d ktiles=%lld per_split=%lld atoms=%d mtiles=%d mt_per_cta=%d "
                 "mranges=%d tmem_cols=%d stages=%d stage_bytes=%d smem=%d grid=(%u,%u,%u) block=%u ws=%zu "
                 "reduce=%s zero=%s out=%s code=%s",
                 ig.halo ? "halo" : "pertap", ig.xs ? "mn" : "m", ig.Nmma, mode, pl.S, ig.cluster, ig.Gm, ig.n_gblocks, ig.n_cchunks, ig.Nt, ig.n_ntiles, ig.n_katoms, ig.box[0], ig.box[1],
                 ig.box[2], ig.box[3], ig.KT, ig.total_kt, pl.per_split, ig.n_atoms, ig.n_mtiles, ig.mt_per_cta,
                 ig.n_mranges, ig.tmem_cols, ig.stages, ig.stage_bytes, ig.smem_bytes, pl.grid[0], pl.grid[1],
                 pl.grid[2], pl.block, pl.ws_bytes,
                 pl.mode == MODE_DETERMINISTIC ? "kernel" : pl.acc_ws ? "cast" : "none",
                 pl.mode == MODE_ATOMIC ? "kernel" : "none", ig.staged ? "staged" : "direct",
                 ig.spec == 2 ? "pair" : ig.spec ? "x1" : "any");
    } else {
        const DwPlan& dw = pl.dw;
        snprintf(buf, sizeof buf,
                 "kernel=depthwise mode=%s S=%d Gm=%d CB=%d cblocks=%d R=%d nseg=%d seg_len=%d threads=%d "
                 "xtile=(w%d,h%d) tiles=%lld per_split=%lld stages=%d stage_bytes=%d smem=%d sliding=%d "
                 "grid=(%u,%u,%u) block=%u ws=%zu reduce=%s zero=%s",
                 mode, pl.S, dw.Gm, dw.CB, dw.n_cblocks, dw.R, dw.nseg, dw.seg_len, dw.threads, dw.xw, dw.xh,
                 dw.total_tiles, pl.per_split, dw.stages, dw.stage_bytes, dw.smem_bytes, dw.sliding, pl.grid[0],
                 pl.grid[1], pl.grid[2], pl.block, pl.ws_bytes,
                 pl.mode == MODE_DETERMINISTIC ? "kernel" : pl.acc_ws ? "cast" : "none",
                 pl.mode == MODE_ATOMIC ? "kernel" : "none");
    }
    (void)pb;
    return buf;
}

namespace {

// Phases of one spatial dim of the backward-data problem (see DgDim).
bool dg_dim(int in, int F, int s, int dil, int pl, DgDim* o, int* span)
{
    if (s > kDgMaxPhases || F > kDgMaxTaps) return false;
    std::memset(o, 0, sizeof *o);
    o->nph = s;
    *span = 0;
    for (int r = 0; r < s; ++r) {
        o->J[r] = in > r ? (int)cdiv(in - r, s) : 0;
        int qmin = 0, qmax = 0, n = 0;
        int q[kDgMaxTaps];
        for (int t = 0; t < F; ++t) {
            const int v = r + pl - t * dil;
            if (((v % s) + s) % s) continue;
            q[t] = (v - ((v % s) + s) % s) / s;  // exact: v is a multiple of s
            if (n == 0 || q[t] < qmin) qmin = q[t];
            if (n == 0 || q[t] > qmax) qmax = q[t];
            o->tap[r][n++] = (unsigned char)t;
        }
        o->ntap[r] = n;
        o->qmin[r] = qmin;
        for (int i = 0; i < n; ++i) o->shift[r][i] = (unsigned char)(q[o->tap[r][i]] - qmin);
        if (n) *span = std::max(*span, qmax - qmin);
    }
    return true;
}

}  // namespace

int make_dgrad_plan(const wg_problem* p, const DeviceCaps& caps, DgPlan* pl, std::string* err)
{
    std::memset(pl, 0, sizeof *pl);
    int st = normalize(p, &pl->pb, err);
    if (st) return st;
    const Problem& pb = pl->pb;
    DgPlan& d = *pl;
    if (((long long)pb.G * pb.K) % 8 || ((long long)pb.G * pb.C) % 8)
        return fail(err, WG_ERR_NOT_SUPPORTED, "backward-data: G*C and G*K must be multiples of 8 (16-byte pixel rows)");
    // Group fold for small C and K: the widest Gm with Gm*C and Gm*K at most 64
    // and multiples of 8 (16-byte rows of the folded W and aligned dY windows).
    d.Gm = 1;
    for (int g = std::min(pb.G, 64); g >= 2; --g)
        if (g * pb.C <= 64 && g * pb.K <= 64 && (g * pb.C) % 8 == 0 && (g * pb.K) % 8 == 0) {
            d.Gm = g;
            break;
        }
    if (d.Gm == 1) {
        if (pb.C % 8) return fail(err, WG_ERR_NOT_SUPPORTED, "backward-data: C must be a multiple of 8 (16-byte W rows)");
        if (pb.G > 1 && pb.K % 8)
            return fail(err, WG_ERR_NOT_SUPPORTED, "backward-data: K must be a multiple of 8 when G > 1");
    }
    d.Gb = (int)cdiv(pb.G, d.Gm);
    d.Cm = d.Gm * pb.C;
    d.Km = d.Gm * pb.K;
    d.ws_bytes = d.Gm > 1 ? (size_t)d.Gb * d.Km * (size_t)pb.T * d.Cm * 2 : 0;
    if (d.Gb > 65535) return fail(err, WG_ERR_NOT_SUPPORTED, "backward-data: too many groups");
    if (pb.ndim == 1) {
        d.bw = 128, d.bh = 1;
    } else {
        d.bw = 8, d.bh = 16;
    }
    int span[3];
    for (int j = 0; j < 3; ++j) {
        // dim[0] = w, dim[1] = h, dim[2] = d; the problem holds (D, H, W).
        const int k = 2 - j;
        if (!dg_dim(pb.in[k], pb.filt[k], pb.stride[k], pb.dil[k], pb.pad_l[k], &d.dim[j], &span[j]))
            return fail(err, WG_ERR_NOT_SUPPORTED, "backward-data: stride above 8 or more than 32 taps along a dim");
    }
    d.PW = d.bw + span[0];
    d.PH = d.bh + span[1];
    if (d.PW > 256 || d.PH > 256)
        return fail(err, WG_ERR_NOT_SUPPORTED, "backward-data: dilated filter too wide for a 256-row patch");
    int mx[3] = {0, 0, 0}, mJ[3] = {0, 0, 0};
    for (int j = 0; j < 3; ++j)
        for (int r = 0; r < d.dim[j].nph; ++r) {
            mx[j] = std::max(mx[j], d.dim[j].ntap[r]);
            mJ[j] = std::max(mJ[j], d.dim[j].J[r]);
        }
    d.max_yx = std::max(1, mx[0] * mx[1]);
    d.patch_bytes = round_up(d.PW * d.PH * 128, 1024);
    d.n_kc = (int)cdiv(d.Km, 64);
    // N-tile and taps per stage: the widest N-tile (up to 128 channels) with
    // every (y, x) tap of a phase's plane in one stage and two stages in shared
    // memory; else 64 channels and the taps in groups.
    const int avail = kMaxSmemPerCta - 2048 - kDgStaging;
    const int cmax = round_up(d.Cm, 16);
    d.Nt = 0;
    // At most 128: two accumulator buffers of 2 Nt columns then leave TMEM room
    // for two CTAs per SM (1x1 stride 2, C 256: 40.8 us against 53.4 us at 256).
    for (int nt = 128; nt >= 16; nt /= 2) {
        if (nt > cmax && nt > 16) continue;
        const int na = (int)cdiv(nt, 64);
        if (2 * (d.patch_bytes + d.max_yx * na * 8192) <= avail) {
            d.Nt = nt;
            d.TG = d.max_yx;
            break;
        }
    }
    if (!d.Nt) {
        d.Nt = std::min(64, cmax);
        d.TG = (avail / 2 - d.patch_bytes) / 8192;
        if (d.TG < 1) return fail(err, WG_ERR_NOT_SUPPORTED, "backward-data: the dY patch does not fit shared memory");
    }
    d.n_catoms = (int)cdiv(d.Nt, 64);
    d.n_ctiles = (int)cdiv(d.Cm, d.Nt);
    // Shared memory: resident W tiles (with a single (channel tile, group) every
    // persistent CTA needs the same W tiles, loaded once) or W streamed with each
    // patch, and a ring that runs on across a CTA's tiles, as deep as fits (<= 4).
    // Two CTAs per SM come first (measured on GB300: two MMA issuers keep the
    // tensor pipe busier than one at N <= 128, e.g. 56x56 C = K = 64: 18.7 us
    // against 22.5 us with one CTA, W resident and a four-deep ring; 1x1
    // stride 2, C 256: 36.9 against 53.5 us); then one CTA per SM, W resident
    // only beside at least three patch stages.
    const long long w_all = (long long)d.n_kc * pb.T * d.n_catoms * 8192;
    const int streamed = d.patch_bytes + d.TG * d.n_catoms * 8192;
    const int half = kMaxSmemPerCta / 2 - 1024 - 2048 - kDgStaging;  // ring + W of one of two CTAs
    const bool tmem_half = pow2_at_least(2 * d.Nt) <= kMaxTmemCols / 2;
    const bool can_res = d.n_ctiles * d.Gb == 1;
    if (tmem_half && can_res && w_all + d.patch_bytes <= half) {
        d.w_resident = 1, d.w_bytes = (int)w_all, d.stage_bytes = d.patch_bytes;
        d.stages = std::min(4, (half - d.w_bytes) / d.stage_bytes);
    } else if (tmem_half && streamed <= half) {
        d.w_resident = 0, d.w_bytes = 0, d.stage_bytes = streamed;
        d.stages = std::min(4, half / d.stage_bytes);
    } else {
        d.w_resident = (can_res && w_all + 3LL * d.patch_bytes <= avail) ? 1 : 0;
        d.w_bytes = d.w_resident ? (int)w_all : 0;
        d.stage_bytes = d.w_resident ? d.patch_bytes : streamed;
        d.stages = std::min(4, (avail - d.w_bytes) / d.stage_bytes);
    }
    d.smem_bytes = d.w_bytes + d.stages * d.stage_bytes + kDgStaging + 2048;
    d.tmem_cols = std::max(32, pow2_at_least(2 * d.Nt));  // two accumulator buffers
    d.n_tw = (int)cdiv(std::max(1, mJ[0]), d.bw);
    d.n_th = (int)cdiv(std::max(1, mJ[1]), d.bh);
    d.n_td = std::max(1, mJ[2]);
    d.n_phases = d.dim[0].nph * d.dim[1].nph * d.dim[2].nph;
    d.n_tiles = (long long)d.n_phases * d.n_tw * d.n_th * d.n_td * pb.N;
    if (d.n_tiles > (1ll << 31) - 1) return fail(err, WG_ERR_NOT_SUPPORTED, "backward-data: too many pixel tiles");
    d.n_all = d.n_tiles * d.n_ctiles * d.Gb;
    if (d.n_all > (1ll << 31) - 1) return fail(err, WG_ERR_NOT_SUPPORTED, "backward-data: too many tiles");
    // Persistent grid: one CTA per SM (two when shared memory and TMEM allow),
    // never more CTAs than tiles.
    const int per_sm = (d.smem_bytes <= kMaxSmemPerCta / 2 - 1024 && d.tmem_cols <= 256) ? 2 : 1;
    d.grid[0] = (unsigned)std::min<long long>(d.n_all, (long long)caps.num_sms * per_sm);
    d.grid[1] = 1;
    d.grid[2] = 1;
    d.block = 192;
    return WG_OK;
}

std::string dgrad_plan_string(const DgPlan& d)
{
    char buf[512];
    snprintf(buf, sizeof buf,
             "kernel=dgrad_tcgen05 Gm=%d w_resident=%d phases=%d box=(w%d,h%d) patch=(w%d,h%d) Nt=%d catoms=%d "
             "ctiles=%d "
             "kchunks=%d max_yx_taps=%d taps/stage=%d patch_bytes=%d stage_bytes=%d ring=%d smem=%d tmem_cols=%d "
             "grid=(%u,%u,%u) block=%u ws=%zu",
             d.Gm, d.w_resident, d.n_phases, d.bw, d.bh, d.PW, d.PH, d.Nt, d.n_catoms, d.n_ctiles, d.n_kc, d.max_yx, d.TG, d.patch_bytes,
             d.stage_bytes, d.stages, d.smem_bytes, d.tmem_cols, d.grid[0], d.grid[1], d.grid[2], d.block,
             d.ws_bytes);
    return buf;
}

}  // namespace wg
