// Host-side problem normalisation and launch planning for the wgrad kernels.
// Pure C++ (no CUDA calls): the plan is a function of the problem, the options
// and the device facts in DeviceCaps.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <string>

#include "../../include/wgrad.h"

namespace wg {

constexpr int kDefaultSMs = 152;        // GB300: 2 dies x 76 SMs
constexpr int kMaxSmemPerCta = 232448;  // 227 KB opt-in dynamic shared memory
constexpr int kMaxTmemCols = 512;
constexpr int kMaxPatches = 32;
constexpr int kMaxMtPerCta = 16;  // M-tiles one CTA accumulates (the kernel's register table size)
constexpr int kMaxHaloAtoms = 256;
constexpr int kMaxHaloFilter = 32;

enum Kind { KIND_IGEMM = 0, KIND_DEPTHWISE = 1 };
enum Mode { MODE_DIRECT = 1, MODE_ATOMIC = 2, MODE_DETERMINISTIC = 3 };

// Normalised problem: every spatial array has 3 entries ordered (D, H, W);
// lower ranks put 1 (pads 0) in the leading unused entries.
struct Problem {
    int ndim, G, N, C, K;
    int in[3], filt[3], out[3], stride[3], dil[3], pad_l[3], pad_r[3];
    int in_dtype, out_dtype;
    long long T;  // filter taps Z*Y*X
    long long P;  // GemmK = N*Do*Ho*Wo
    long long x_elems, dy_elems, dw_elems;
};

// Tensor-core implicit GEMM (kernel igemm_wgrad).  The CTA tile is
// D[(tap, c) rows x k cols]; rows come in "atoms" of 64 channels of one tap.
struct IgemmPlan {
    int Gm;           // groups folded into one CTA channel window
    int n_gblocks;    // ceil(G / Gm)
    int n_cchunks;    // 64-channel chunks per tap in the window
    int Nt;           // MMA N (k columns per N-tile), multiple of 16, <= 256
    int n_ntiles;     // N-tiles over the k window
    int n_katoms;     // 64-wide dY chunks per N-tile
    int box[4];       // pixel tile extent along (w, h, d, n)
    int ntile[4];     // tiles along (w, h, d, n)
    int KT;           // pixels per K-tile = product of box
    long long total_kt;
    int n_atoms;      // taps x chunks
    int n_mtiles;     // ceil(n_atoms / 2): MMA M = 128 = two atoms
    int mt_per_cta;   // M-tiles accumulated by one CTA (TMEM columns = mt_per_cta * Nt)
    int n_mranges;    // ceil(n_mtiles / mt_per_cta)
    int tmem_cols;    // power of two >= mt_per_cta * Nt
    int stages;
    int slot_bytes;   // KT * 128 bytes: one 64-channel dY chunk of one K-tile
    int stage_bytes;
    int smem_bytes;   // dynamic shared memory per CTA
    // X staging.  halo = 1: per K-tile one patch per (stride phase, channel
    // chunk) covering every tap, taps read as row-shifted views of it.
    // halo = 0: one box per atom (tap, chunk), 2 * mt_per_cta boxes per K-tile.
    int halo;
    int patch[3];     // patch extent along (w, h, d) in strided input pixels
    int patch_bytes;  // bytes per patch, 1024-aligned
    int n_patches;    // patches (or boxes) per K-tile
    int dy_off;       // byte offset of the dY chunks inside a stage
    int n_phase[3];   // stride phases used along (w, h, d)
    unsigned char patch_ph[kMaxPatches][4];  // phase value (w, h, d) and channel chunk of each patch
    unsigned int atom_off[kMaxHaloAtoms];    // byte offset of atom (patch + tap row shift) in a stage
    unsigned short atom_tap[kMaxHaloAtoms];
    unsigned char atom_cc[kMaxHaloAtoms];
    // Tap form.  xs = 0: every tap on the MMA rows, atoms are (tap, chunk).
    // xs = X (2..4): the filter's x taps on the MMA columns.  Atoms are
    // (z, y, chunk) rows of an X patch with no halo along w; the B operand is
    // one dY patch per K-tile, dy_w = box w + (X-1)*dil_w columns wide, read
    // as xs 64-column atoms (atom j = tap x = X-1-j, a row shift of j*dil_w),
    // so the MMA N is Nmma = 64*xs.  Pixel tiles run over q = wo + x*dil_w in
    // [0, Wo + (X-1)*dil_w) along w; dY is zero outside [0, Wo) (TMA fill).
    int xs;
    int Nmma;         // MMA N (Nt when xs = 0)
    int dy_w;         // dY staging extent along w (box w when xs = 0)
    int dy_bytes;     // dY bytes per stage (the TMA transaction count of its boxes)
    long long est_cycles;  // planner's cost estimate (for the plan string)
    long long tile_clk;    // planner's estimate of one K-tile on one CTA, in SM cycles
    int cluster;           // CTAs per thread-block cluster along the split (1: none)
    int staged;            // 1: each CTA's results are one contiguous dW block, written from shared memory
    int spec;              // kernel instance: 2 = the CTA pair; 1 = x taps on the columns, one M-tile per CTA, split mode; 0 = any plan
    // CTA pair (xs > 0, two M-tiles): the M-tiles of a split run on the two
    // CTAs of a cluster that share M = 256 MMAs (tcgen05 .cta_group::2); each
    // stages 32 of the 64 output channels of the dY patch (dy_bytes is that
    // half, at offset 0 of the stage) and the same X patch, rank 0's at
    // pair_xoff and rank 1's pair_xshift bytes lower (the row offset of atom
    // 2), so that one A descriptor serves both.
    int pair, pair_xoff, pair_xshift;
};

// CUDA-core depthwise kernel (cpg = kpg = 1).
struct DwPlan {
    int CB;           // channels per CTA
    int n_cblocks;
    int Gm;           // channels per thread vector (group-merge degree)
    int R;            // output rows per tile
    int nseg;         // column segments per row
    int seg_len;      // output columns per segment
    int threads;      // compute threads (a producer warp is added on top)
    int xw, xh;       // X tile extent (w, h) in input pixels
    long long total_tiles;  // N * ceil(Ho / R)
    int stages;
    int x_bytes, dy_bytes, stage_bytes, smem_bytes;
    int sliding;      // 1: register sliding window along W (stride 1, dilation 1 in W)
};

// Split-K workspace (deterministic mode): dW viewed as ws_rows rows of ws_L
// elements, each row cut into ws_nj slices of ws_W elements; the n_out
// partials of a slice are stored together (see WsLayout in ptx.cuh).
struct Plan {
    Problem pb;
    int kind;
    int mode;
    int S;              // split degree of GemmK
    // Atomic mode with a 16-bit dW: the splits add into an fp32 copy of dW in
    // the workspace (zeroed first), which a cast kernel then converts to dW.
    int acc_ws;
    long long per_split;  // K-tiles (igemm) or row tiles (depthwise) per split
    int n_out;          // partial sums per dW element that reach memory (S / cluster)
    long long ws_rows, ws_L;
    int ws_W, ws_nj;
    size_t ws_bytes;
    unsigned grid[3];
    unsigned block;
    IgemmPlan ig;
    DwPlan dw;
};

// Validate and normalise.  Returns a wg_status; *err gets the reason.
int normalize(const wg_problem* p, Problem* out, std::string* err);

// Device facts the planner uses: SM count and, for clusters of 1, 2, 4 and 8
// CTAs of the tensor-core kernel at its largest shared-memory size, how many
// CTAs fit on the device at once (clusters must sit within one GPC).
struct DeviceCaps {
    int num_sms;
    int cluster_ctas[4];
};

// GB300 values (measured), used when no device can be queried.
DeviceCaps default_caps(int num_sms);

// Choose kernel, tiles, split degree, cluster size and mode.
int make_plan(const wg_problem* p, const wg_options* opt, const DeviceCaps& caps, Plan* out, std::string* err);

std::string plan_string(const Plan& pl);

// Backward-data (dgrad) on the tensor cores: dX[pixel, c] = sum over (k, tap)
// of dY[pixel shifted by the tap, k] * W[k, tap, c].  A CTA owns a box of 128
// input pixels of one image and depth slice (8 x 16, or 128 along W for 1-D
// problems), an N-tile of C and one group; it walks (K chunk of 64, filter
// plane z, tap group) stages, each a dY halo patch (one row-shifted view per
// tap) plus the W tiles of the group's taps.
// Strides: the input positions of one dim split into `stride` phases
// i = r + stride * j.  In phase r only the taps t with (r + pad_l - t*dil)
// divisible by the stride contribute, each reading dY at j + q_t,
// q_t = (r + pad_l - t*dil) / stride; per phase the taps are listed with their
// row shift q_t - min q.  Stride 1 is the single phase r = 0 with every tap.
constexpr int kDgMaxPhases = 8;
constexpr int kDgStaging = 8192;  // epilogue staging of the backward-data kernel (4 warps x 32 x 64 B)
constexpr int kDgMaxTaps = 32;
struct DgDim {
    int nph;                                          // phases (= stride)
    int J[kDgMaxPhases];                              // positions in each phase
    int qmin[kDgMaxPhases];                           // dY offset of the phase's first patch row
    int ntap[kDgMaxPhases];                           // contributing taps
    unsigned char tap[kDgMaxPhases][kDgMaxTaps];      // their filter index
    unsigned char shift[kDgMaxPhases][kDgMaxTaps];    // their row shift in the patch
};

struct DgPlan {
    Problem pb;
    // Group fold: Gm groups with small C and K share one tile; the kernel sees
    // Gb = ceil(G / Gm) "groups" of Cm = Gm*C and Km = Gm*K channels and reads
    // a block-diagonal copy of W (zero between different groups), written into
    // the workspace by an expansion kernel.  Gm = 1: W is read as it is.
    int Gm, Gb, Cm, Km;
    size_t ws_bytes;      // the block-diagonal W (0 when Gm = 1)
    int bw, bh;           // pixel box along (w, h), in phase positions
    int PW, PH;           // dY patch extent along (w, h)
    int Nt, n_catoms, n_ctiles;
    int n_kc;             // 64-channel chunks of K
    int TG;               // taps per stage (of one plane's (y, x) taps)
    int max_yx;           // most (y, x) taps of any phase
    int patch_bytes;      // dY patch bytes (1024-aligned)
    int w_resident;       // 1: one (channel tile, group) and all its W tiles fit: loaded once per CTA
    int w_bytes;          // resident W bytes (0 when streamed with the patches)
    int stage_bytes, stages, smem_bytes, tmem_cols;
    int n_tw, n_th, n_td; // boxes along w and h, depth positions, per phase (the largest phase)
    int n_phases;         // nph_w * nph_h * nph_d
    long long n_tiles;    // n_phases * n_tw * n_th * n_td * N
    long long n_all;      // n_tiles * n_ctiles * Gb: the persistent CTAs' tile list
    DgDim dim[3];         // (w, h, d)
    unsigned grid[3];
    unsigned block;
};

int make_dgrad_plan(const wg_problem* p, const DeviceCaps& caps, DgPlan* out, std::string* err);

std::string dgrad_plan_string(const DgPlan& pl);

}  // namespace wg
