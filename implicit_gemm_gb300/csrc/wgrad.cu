// C ABI of libwgrad.so (declared in include/wgrad.h): validation, planning,
// TMA tensor-map encoding and kernel launches.  No device memory is allocated
// here; every buffer is the caller's.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <string>

#include "../../include/wgrad.h"
#include "k_depthwise.cuh"
#include "k_dgrad.cuh"
#include "k_igemm.cuh"
#include "k_igemm_pair.cuh"
#include "plan.h"

static_assert(wg::kDgStaging == wg::kDgStagingBytes, "planner and kernel disagree on the dgrad staging size");

namespace wg {

// One thread waits on an mbarrier that nothing completes: the bounded wait
// runs out, sets the status word and returns (wg_selftest_timeout).
__global__ void selftest_timeout_kernel()
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
        (void)mbar_wait(&bar, 0);
    }
}

}  // namespace wg

namespace {

thread_local std::string g_err;
// Event recorded after each call's main kernel (wg_set_mark_event); null = off.
thread_local cudaEvent_t g_mark = nullptr;

int set_err(int status, const std::string& msg)
{
    g_err = msg;
    return status;
}

int cuda_fail(const char* what, cudaError_t e)
{
    return set_err(WG_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// Raise a kernel's dynamic shared-memory limit when a launch needs more than
// any earlier one (per device).
template <typename K>
int ensure_smem(K kernel, int bytes)
{
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> done;
    int dev = 0;
    cudaGetDevice(&dev);
    const auto key = std::make_pair(reinterpret_cast<const void*>(kernel), dev);
    std::lock_guard<std::mutex> lk(mu);
    auto it = done.find(key);
    if (it != done.end() && it->second >= bytes) return WG_OK;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return cuda_fail("cudaFuncSetAttribute", e);
    done[key] = bytes;
    return WG_OK;
}

// SM count of the current device (kDefaultSMs when no device is visible, so
// host-only queries give the same plan on a machine without a GPU).
int num_sms()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return wg::kDefaultSMs;
    }
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return wg::kDefaultSMs;
    }
    return n;
}

// Device facts for the planner: SM count, and how many CTAs of the
// tensor-core kernel (at its largest shared-memory size) fit at once in
// clusters of 1, 2, 4 and 8, from the occupancy calculator.  Queried once per
// device; GB300 defaults when there is no device.
wg::DeviceCaps device_caps()
{
    static std::mutex mu;
    static std::map<int, wg::DeviceCaps> cache;
    const int sms = num_sms();
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return wg::default_caps(sms);
    }
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    wg::DeviceCaps c = wg::default_caps(sms);
    const int smem = wg::kMaxSmemPerCta;
    if (ensure_smem(wg::igemm_wgrad_kernel<0>, smem) == WG_OK) {
        for (int i = 0, q = 1; i < 4; ++i, q *= 2) {
            cudaLaunchConfig_t cfg = {};
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 1;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = (unsigned)q;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            cfg.gridDim = dim3(1, 1, (unsigned)q);
            cfg.blockDim = dim3(wg::kIgThreads);
            cfg.dynamicSmemBytes = (size_t)smem;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, wg::igemm_wgrad_kernel<0>, &cfg) == cudaSuccess && n > 0)
                c.cluster_ctas[i] = n * q;
            else
                cudaGetLastError();
        }
    } else {
        cudaGetLastError();
    }
    cache.emplace(dev, c);
    return c;
}

// Plans are a pure function of (problem, options, device facts); successful
// ones are cached so that repeated calls skip the tile search.
int plan_for(const wg_problem* p, const wg_options* opt, wg::Plan* pl, std::string* key_out = nullptr)
{
    static std::mutex mu;
    static std::map<std::string, wg::Plan> cache;
    const wg::DeviceCaps caps = device_caps();
    std::string key;
    if (p) {
        wg_options o{0, WG_MODE_AUTO, 0, 0, WG_KERNEL_AUTO};
        if (opt) o = *opt;
        key.assign(reinterpret_cast<const char*>(p), sizeof *p);
        key.append(reinterpret_cast<const char*>(&o), sizeof o);
        key.append(reinterpret_cast<const char*>(&caps), sizeof caps);
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *pl = it->second;
            if (key_out) *key_out = key;
            return WG_OK;
        }
    }
    std::string err;
    const int st = wg::make_plan(p, opt, caps, pl, &err);
    if (st) return set_err(st, err);
    std::lock_guard<std::mutex> lk(mu);
    if (cache.size() > 1024) cache.clear();
    cache.emplace(key, *pl);
    if (key_out) *key_out = key;
    return WG_OK;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

int encode(CUtensorMap* tm, int in_dtype, void* base, const cuuint64_t dims[5], const cuuint32_t box[5],
           const cuuint32_t estr[5], CUtensorMapSwizzle swz, const char* what)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return set_err(WG_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    cuuint64_t strides[4];
    cuuint64_t s = dims[0] * 2;
    for (int i = 0; i < 4; ++i) {
        strides[i] = s;
        s *= dims[i + 1];
    }
    const CUtensorMapDataType dt = in_dtype == WG_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUresult r = fn(tm, dt, 5, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char buf[256];
        snprintf(buf, sizeof buf, "cuTensorMapEncodeTiled(%s) failed with CUresult %d (box %u,%u,%u,%u,%u)", what, (int)r,
                 box[0], box[1], box[2], box[3], box[4]);
        return set_err(WG_ERR_CUDA, buf);
    }
    return WG_OK;
}

wg::WsLayout ws_layout(const wg::Plan& pl)
{
    wg::WsLayout w;
    w.L = pl.ws_L;
    w.W = pl.ws_W;
    w.nj = pl.ws_nj;
    w.S = pl.n_out;
    return w;
}

// Encoded tensor maps and kernel parameters of one (plan, buffers) pair, kept
// so that a repeated call only launches.
struct Prepared {
    CUtensorMap tmx, tmy;
    wg::IgParams ig;
    wg::DwParams dw;
};

std::mutex g_prep_mu;
std::map<std::string, Prepared>& prep_cache()
{
    static std::map<std::string, Prepared> m;
    return m;
}

std::string prep_key(const std::string& plan_key, const void* x, const void* dy, const void* dw, const void* ws)
{
    int dev = 0;
    cudaGetDevice(&dev);
    const void* ptrs[4] = {x, dy, dw, ws};
    std::string k = plan_key;
    k.append(reinterpret_cast<const char*>(ptrs), sizeof ptrs);
    k.append(reinterpret_cast<const char*>(&dev), sizeof dev);
    return k;
}

int prepare_igemm(const wg::Plan& pl, const void* x, const void* dy, void* dw, void* ws, Prepared* out)
{
    const wg::Problem& pb = pl.pb;
    const wg::IgemmPlan& ig = pl.ig;
    CUtensorMap& tmx = out->tmx;
    CUtensorMap& tmy = out->tmy;
    const cuuint64_t GC = (cuuint64_t)pb.G * pb.C, GK = (cuuint64_t)pb.G * pb.K;
    {
        const cuuint64_t dims[5] = {GC, (cuuint64_t)pb.in[2], (cuuint64_t)pb.in[1], (cuuint64_t)pb.in[0],
                                    (cuuint64_t)pb.N};
        const cuuint32_t box[5] = {64, (cuuint32_t)(ig.patch[0] * pb.stride[2]), (cuuint32_t)(ig.patch[1] * pb.stride[1]),
                                   (cuuint32_t)(ig.patch[2] * pb.stride[0]), (cuuint32_t)ig.box[3]};
        const cuuint32_t estr[5] = {1, (cuuint32_t)pb.stride[2], (cuuint32_t)pb.stride[1], (cuuint32_t)pb.stride[0], 1};
        const int st = encode(&tmx, pb.in_dtype, const_cast<void*>(x), dims, box, estr, CU_TENSOR_MAP_SWIZZLE_128B, "X");
        if (st) return st;
    }
    {
        const cuuint64_t dims[5] = {GK, (cuuint64_t)pb.out[2], (cuuint64_t)pb.out[1], (cuuint64_t)pb.out[0],
                                    (cuuint64_t)pb.N};
        // A CTA of a pair stages 32 output channels (64-byte rows, 64-byte swizzle).
        const cuuint32_t box[5] = {ig.pair ? 32u : 64u, (cuuint32_t)ig.dy_w, (cuuint32_t)ig.box[1],
                                   (cuuint32_t)ig.box[2], (cuuint32_t)ig.box[3]};
        const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        const int st = encode(&tmy, pb.in_dtype, const_cast<void*>(dy), dims, box, estr,
                              ig.pair ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, "dY");
        if (st) return st;
    }
    wg::IgParams& prm = out->ig;
    memset(&prm, 0, sizeof prm);
    prm.G = pb.G, prm.C = pb.C, prm.K = pb.K, prm.T = (int)pb.T, prm.GC = (int)GC, prm.GK = (int)GK;
    prm.X = pb.filt[2], prm.Y = pb.filt[1];
    prm.ncc = ig.n_cchunks;
    for (int i = 0; i < 3; ++i) {
        prm.s[i] = pb.stride[2 - i];
        prm.d[i] = pb.dil[2 - i];
        prm.pl[i] = pb.pad_l[2 - i];
        prm.patch[i] = ig.patch[i];
    }
    for (int i = 0; i < 4; ++i) prm.box[i] = ig.box[i], prm.ntile[i] = ig.ntile[i];
    prm.KT = ig.KT, prm.ksteps = ig.KT / 16;
    prm.per_split = (int)pl.per_split, prm.total_kt = (int)ig.total_kt;
    prm.Gm = ig.Gm, prm.Nt = ig.Nt, prm.n_ntiles = ig.n_ntiles, prm.n_katoms = ig.n_katoms;
    prm.n_atoms = ig.n_atoms, prm.n_mtiles = ig.n_mtiles, prm.mtpc = ig.mt_per_cta;
    prm.halo = ig.halo;
    prm.xs = ig.xs, prm.Nmma = ig.Nmma, prm.dy_tx = ig.dy_bytes;
    prm.dy_xoff = ig.xs ? (pb.filt[2] - 1) * pb.dil[2] : 0;
    prm.patch_bytes = ig.patch_bytes;
    prm.patch_tx = ig.halo ? ig.patch[0] * ig.patch[1] * ig.patch[2] * ig.box[3] * 128 : ig.slot_bytes;
    prm.n_patches = ig.n_patches, prm.dy_off = ig.dy_off, prm.slot_bytes = ig.slot_bytes;
    prm.stage_bytes = ig.stage_bytes, prm.stages = ig.stages, prm.tmem_cols = ig.tmem_cols;
    prm.idesc = wg::make_idesc_f16(pb.in_dtype == WG_BF16, true, true, ig.pair ? 256 : 128, ig.Nmma);
    prm.pair = ig.pair, prm.pair_xoff = ig.pair_xoff, prm.pair_xshift = ig.pair_xshift;
    prm.mode = pl.mode, prm.out_dtype = pb.out_dtype;
    prm.clq = ig.cluster;
    prm.staged = ig.staged;
    if (ig.staged) {
        // Inverse atom table: (tap / X, chunk) -> atom index (x = 0 taps when
        // the x taps sit on the columns; every atom when they do not).
        const int xe = ig.xs ? ig.xs : 1;
        for (int i = 0; i < ig.n_atoms; ++i) {
            const int tap = ig.halo ? ig.atom_tap[i] : i / ig.n_cchunks;
            const int cc = ig.halo ? ig.atom_cc[i] : i % ig.n_cchunks;
            prm.atom_of[(tap / xe) * ig.n_cchunks + cc] = (unsigned char)i;
        }
    }
    prm.out = pl.mode == wg::MODE_DETERMINISTIC || pl.acc_ws ? ws : dw;
    prm.ws = ws_layout(pl);
    // K-step descriptor parts: pixel row r of the tile (w fastest) sits at patch
    // row ((in*PD + id)*PH + ih)*PW + iw of a halo patch, at row r of a per-tap box.
    for (int ks = 0; ks < 16 && ks < ig.KT / 16; ++ks) {
        unsigned r[2];
        for (int h = 0; h < 2; ++h) {
            int q = 16 * ks + 8 * h;
            const int iw = q % ig.box[0];
            q /= ig.box[0];
            const int ih = q % ig.box[1];
            q /= ig.box[1];
            const int id = q % ig.box[2];
            const int in = q / ig.box[2];
            r[h] = ig.halo ? (unsigned)(((in * ig.patch[2] + id) * ig.patch[1] + ih) * ig.patch[0] + iw)
                           : (unsigned)(16 * ks + 8 * h);
        }
        prm.kd_table[ks] = ((unsigned long long)((r[1] - r[0]) * 8u) << 32) + (unsigned long long)(r[0] * 8u);
        if (ig.xs) {
            // B: the same pixels in the dY patch, dy_w rows per (n, d, h) row.
            for (int h = 0; h < 2; ++h) {
                int q = 16 * ks + 8 * h;
                const int iw = q % ig.box[0];
                q /= ig.box[0];
                const int ih = q % ig.box[1];
                q /= ig.box[1];
                const int id = q % ig.box[2];
                const int in = q / ig.box[2];
                r[h] = (unsigned)(((in * ig.box[2] + id) * ig.box[1] + ih) * ig.dy_w + iw);
            }
            // Rows of 128 bytes (eight 16-byte units), or 64 for a CTA pair's half.
            const unsigned u = ig.pair ? 4u : 8u;
            prm.kd_table_b[ks] =
                ((unsigned long long)((r[1] - r[0]) * u) << 32) + (unsigned long long)(r[0] * u);
        }
    }
    if (ig.halo) {
        memcpy(prm.patch_ph, ig.patch_ph, sizeof prm.patch_ph);
        for (int i = 0; i < ig.n_atoms; ++i) {
            prm.atom_off[i] = ig.atom_off[i];
            prm.atom_tap[i] = ig.atom_tap[i];
            prm.atom_cc[i] = ig.atom_cc[i];
        }
    }
    return WG_OK;
}

// Resident CTAs per SM of the register-path reduction kernel (occupancy
// calculator, once per device).
int reduce_regs_ctas_per_sm()
{
    static std::mutex mu;
    static std::map<int, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 1;
    }
    std::lock_guard<std::mutex> lk(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, wg::reduce_splits_regs_kernel, 128, 0) != cudaSuccess ||
        n <= 0) {
        cudaGetLastError();
        n = 1;
    }
    cache.emplace(dev, n);
    return n;
}

// Programmatic stream serialization for a launch (see launch_pre).
void pdl_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, unsigned* na, cudaStream_t stream)
{
    attr[*na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[*na].val.programmaticStreamSerializationAllowed = 1;
    ++*na;
    cfg->attrs = attr;
    cfg->numAttrs = *na;
    cfg->stream = stream;
}

// Stage 2 of deterministic split-K, launched as a programmatic dependent of the
// split-K kernel just before it on the stream.
int launch_reduce(const wg::Plan& pl, void* ws, void* dw, cudaStream_t stream)
{
    const wg::Problem& pb = pl.pb;
    const wg::WsLayout w = ws_layout(pl);
    // A CTA takes spc consecutive slices (S partial rows of W each, contiguous,
    // plus their range sums): enough that its 256 threads have work when slices
    // are small, while at least four CTAs per SM remain (measured on the 3-D
    // stride-2 workload: 18.4 us per step with four, 20.6 with two, 20.0 with
    // sixteen, 19.4 with one slice per CTA).
    const long long n_slices = pl.ws_rows * w.nj;
    const long long items = (long long)(w.W / 4) * wg::red_groups(w.S);
    long long spc = std::max(1LL, std::min<long long>(16, wg::kRedThreads / std::max(1LL, items)));
    spc = std::max(1LL, std::min(spc, n_slices / (4LL * num_sms())));
    auto smem_for = [&](long long k) { return k * (w.S + wg::kRedGroups) * w.W * 4 + 128; };
    while (spc > 1 && smem_for(spc) > wg::kMaxSmemPerCta) --spc;
    const long long smem = smem_for(spc);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    unsigned na = 0;
    pdl_config(&cfg, attr, &na, stream);
    cfg.blockDim = dim3(wg::kRedThreads);
    cudaError_t e;
    const float* wsf = static_cast<const float*>(ws);
    // Register path when every slice gets its own resident CTA (one wave): all
    // loads of a split range are then in flight at once.  Otherwise the bulk
    // path, which packs several slices per CTA.  Measured: 56x56 two-stage
    // S = 75 (384 slices) 19.5 -> 18.5 us per call, grouped two-stage (256
    // slices) 19.8 -> 18.9 us; 3-D S = 8 (2,592 slices, about six waves of the
    // register kernel) 19.5 us with the bulk path against 22.6 us.
    if (n_slices < (1LL << 31) && w.W <= 128 && n_slices <= (long long)num_sms() * reduce_regs_ctas_per_sm()) {
        cfg.gridDim = dim3((unsigned)n_slices);
        cfg.blockDim = dim3(128);
        e = cudaLaunchKernelEx(&cfg, wg::reduce_splits_regs_kernel, wsf, dw, w, pb.out_dtype);
    } else if (smem <= wg::kMaxSmemPerCta && n_slices < (1LL << 31) && w.W <= 128) {
        const int st = ensure_smem(wg::reduce_splits_bulk_kernel, (int)smem);
        if (st) return st;
        cfg.gridDim = dim3((unsigned)((n_slices + spc - 1) / spc));
        cfg.dynamicSmemBytes = (size_t)smem;
        e = cudaLaunchKernelEx(&cfg, wg::reduce_splits_bulk_kernel, wsf, dw, w, pb.out_dtype, (int)spc, n_slices);
    } else {
        cfg.gridDim = dim3((unsigned)((pb.dw_elems + wg::kRedThreads - 1) / wg::kRedThreads));
        e = cudaLaunchKernelEx(&cfg, wg::reduce_splits_kernel, wsf, dw, pb.dw_elems, w, pb.out_dtype);
    }
    if (e != cudaSuccess) return cuda_fail("reduce_splits launch", e);
    return WG_OK;
}

// A call runs as launch_pre (zero dW, or its fp32 copy in the workspace, for
// atomic accumulation), the main kernel (launch_main), then launch_post (the
// mark event, then the split reduction or the cast of the fp32 copy).
// The zeroing is a kernel of this library rather than cudaMemsetAsync: the main
// kernel is launched as its programmatic dependent and waits for it only
// before its atomic adds (a memset before the main kernel measured ~4 us per
// call on GB300, a dependent zeroing kernel is hidden behind the main loop).
//
// Every kernel of a call is launched with programmatic stream serialization,
// the first one too: it may be scheduled while the kernel before it on the
// stream (the previous call's last kernel, or the caller's) is still running,
// and waits for it (griddepcontrol.wait) before it touches memory that kernel
// may write; its launch and set-up (barriers, tensor-map prefetch) overlap
// that kernel's tail.  A kernel before it that was not launched this way, or
// a copy or event between them, gives ordinary stream order.
int launch_pre(const wg::Plan& pl, void* ws, void* dw, cudaStream_t stream)
{
    if (pl.mode == wg::MODE_ATOMIC) {
        // The adds go to dW, or (16-bit dW) to its fp32 copy in the workspace.
        float* acc = static_cast<float*>(pl.acc_ws ? ws : dw);
        const long long n = pl.pb.dw_elems;
        const long long blocks = std::max(1LL, std::min<long long>((n / 4 + 255) / 256, 4LL * num_sms()));
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        unsigned na = 0;
        pdl_config(&cfg, attr, &na, stream);
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(256);
        const cudaError_t e = cudaLaunchKernelEx(&cfg, wg::zero_f32_kernel, acc, n);
        if (e != cudaSuccess) return cuda_fail("zero_f32_kernel launch", e);
    }
    return WG_OK;
}

int launch_igemm_main(const wg::Plan& pl, const Prepared& pr, cudaStream_t stream)
{
    const wg::IgemmPlan& ig = pl.ig;
    auto kernel = ig.spec == 2   ? wg::igemm_wgrad_pair_kernel
                  : ig.spec == 1 ? wg::igemm_wgrad_kernel<1>
                                 : wg::igemm_wgrad_kernel<0>;
    const int st = ensure_smem(kernel, ig.smem_bytes);
    if (st) return st;
    // Consecutive splits form a cluster (grid z is a multiple of the cluster
    // size), or the two M-ranges of a split do (CTA pair: grid x = 2); the
    // kernel is a programmatic dependent of the kernel before it (the zeroing
    // kernel in atomic mode).
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (ig.pair) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 2;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    } else if (ig.cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = (unsigned)ig.cluster;
        ++na;
    }
    pdl_config(&cfg, attr, &na, stream);
    cfg.gridDim = dim3(pl.grid[0], pl.grid[1], pl.grid[2]);
    cfg.blockDim = dim3(pl.block);
    cfg.dynamicSmemBytes = (size_t)ig.smem_bytes;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, pr.tmx, pr.tmy, pr.ig);
    if (e != cudaSuccess) return cuda_fail("igemm_wgrad_kernel launch", e);
    return WG_OK;
}

int launch_post(const wg::Plan& pl, void* ws, void* dw, cudaStream_t stream)
{
    if (g_mark) {
        const cudaError_t e = cudaEventRecord(g_mark, stream);
        if (e != cudaSuccess) return cuda_fail("cudaEventRecord(mark)", e);
    }
    if (pl.mode == wg::MODE_DETERMINISTIC) return launch_reduce(pl, ws, dw, stream);
    if (pl.acc_ws) {
        const long long n = pl.pb.dw_elems;
        const long long blocks = std::max(1LL, std::min<long long>((n / 4 + 255) / 256, 4LL * num_sms()));
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        unsigned na = 0;
        pdl_config(&cfg, attr, &na, stream);
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(256);
        const float* src = static_cast<const float*>(ws);
        const cudaError_t e =
            pl.pb.out_dtype == WG_BF16
                ? cudaLaunchKernelEx(&cfg, wg::cast_f32_kernel<__nv_bfloat16>, src, static_cast<__nv_bfloat16*>(dw), n)
                : cudaLaunchKernelEx(&cfg, wg::cast_f32_kernel<__half>, src, static_cast<__half*>(dw), n);
        if (e != cudaSuccess) return cuda_fail("cast_f32_kernel launch", e);
    }
    return WG_OK;
}

template <bool BF16, int GM, bool SLIDE>
int launch_dw_t(const wg::Plan& pl, dim3 grid, const CUtensorMap& tmx, const CUtensorMap& tmy, const wg::DwParams& prm,
                cudaStream_t stream)
{
    auto k = wg::depthwise_wgrad_kernel<BF16, GM, SLIDE>;
    const int st = ensure_smem(k, pl.dw.smem_bytes);
    if (st) return st;
    // A programmatic dependent of the kernel before it (the kernel that zeroes
    // dW in atomic mode).
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    unsigned na = 0;
    pdl_config(&cfg, attr, &na, stream);
    cfg.gridDim = grid;
    cfg.blockDim = dim3(pl.block);
    cfg.dynamicSmemBytes = (size_t)pl.dw.smem_bytes;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, k, tmx, tmy, prm);
    if (e != cudaSuccess) return cuda_fail("depthwise_wgrad_kernel launch", e);
    return WG_OK;
}

template <bool BF16, int GM>
int launch_dw_g(const wg::Plan& pl, dim3 g, const CUtensorMap& a, const CUtensorMap& b, const wg::DwParams& prm,
                cudaStream_t s)
{
    const bool slide = pl.dw.sliding && pl.pb.filt[1] == 3 && pl.pb.filt[2] == 3;
    return slide ? launch_dw_t<BF16, GM, true>(pl, g, a, b, prm, s) : launch_dw_t<BF16, GM, false>(pl, g, a, b, prm, s);
}

template <bool BF16>
int launch_dw_b(const wg::Plan& pl, dim3 g, const CUtensorMap& a, const CUtensorMap& b, const wg::DwParams& prm,
                cudaStream_t s)
{
    switch (pl.dw.Gm) {
        case 1: return launch_dw_g<BF16, 1>(pl, g, a, b, prm, s);
        case 2: return launch_dw_g<BF16, 2>(pl, g, a, b, prm, s);
        case 4: return launch_dw_g<BF16, 4>(pl, g, a, b, prm, s);
        default: return launch_dw_g<BF16, 8>(pl, g, a, b, prm, s);
    }
}

int prepare_depthwise(const wg::Plan& pl, const void* x, const void* dy, void* dw, void* ws, Prepared* out)
{
    const wg::Problem& pb = pl.pb;
    const wg::DwPlan& d = pl.dw;
    CUtensorMap& tmx = out->tmx;
    CUtensorMap& tmy = out->tmy;
    {
        const cuuint64_t dims[5] = {(cuuint64_t)pb.G, (cuuint64_t)pb.in[2], (cuuint64_t)pb.in[1], 1, (cuuint64_t)pb.N};
        const cuuint32_t box[5] = {(cuuint32_t)d.CB, (cuuint32_t)d.xw, (cuuint32_t)d.xh, 1, 1};
        const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        const int st = encode(&tmx, pb.in_dtype, const_cast<void*>(x), dims, box, estr, CU_TENSOR_MAP_SWIZZLE_NONE, "X");
        if (st) return st;
    }
    {
        const cuuint64_t dims[5] = {(cuuint64_t)pb.G, (cuuint64_t)pb.out[2], (cuuint64_t)pb.out[1], 1, (cuuint64_t)pb.N};
        const cuuint32_t box[5] = {(cuuint32_t)d.CB, (cuuint32_t)pb.out[2], (cuuint32_t)d.R, 1, 1};
        const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        const int st = encode(&tmy, pb.in_dtype, const_cast<void*>(dy), dims, box, estr, CU_TENSOR_MAP_SWIZZLE_NONE, "dY");
        if (st) return st;
    }
    wg::DwParams& prm = out->dw;
    memset(&prm, 0, sizeof prm);
    prm.G = pb.G, prm.Ho = pb.out[1], prm.Wo = pb.out[2], prm.Y = pb.filt[1], prm.X = pb.filt[2], prm.T = (int)pb.T;
    prm.sh = pb.stride[1], prm.sw = pb.stride[2], prm.dh = pb.dil[1], prm.dw = pb.dil[2];
    prm.plh = pb.pad_l[1], prm.plw = pb.pad_l[2];
    prm.CB = d.CB, prm.R = d.R, prm.nseg = d.nseg, prm.seg_len = d.seg_len;
    prm.nused = (d.CB / d.Gm) * d.R * d.nseg;
    prm.xw = d.xw, prm.xh = d.xh;
    prm.n_hstrips = (pb.out[1] + d.R - 1) / d.R;
    prm.per_split = (int)pl.per_split, prm.total_tiles = (int)d.total_tiles;
    prm.stages = d.stages, prm.stage_bytes = d.stage_bytes;
    prm.x_bytes_al = (d.x_bytes + 127) / 128 * 128;
    prm.x_tx = d.x_bytes, prm.dy_tx = d.dy_bytes;
    prm.mode = pl.mode, prm.out_dtype = pb.out_dtype;
    prm.out = pl.mode == wg::MODE_DETERMINISTIC || pl.acc_ws ? ws : dw;
    prm.ws = ws_layout(pl);
    return WG_OK;
}

int launch_depthwise_main(const wg::Plan& pl, const Prepared& pr, cudaStream_t stream)
{
    const dim3 grid(pl.grid[0], pl.grid[1], pl.grid[2]);
    return pl.pb.in_dtype == WG_BF16 ? launch_dw_b<true>(pl, grid, pr.tmx, pr.tmy, pr.dw, stream)
                                     : launch_dw_b<false>(pl, grid, pr.tmx, pr.tmy, pr.dw, stream);
}

int launch_call(const wg::Plan& pl, const Prepared& pr, void* dw, void* ws, cudaStream_t stream)
{
    int st = launch_pre(pl, ws, dw, stream);
    if (!st)
        st = pl.kind == wg::KIND_IGEMM ? launch_igemm_main(pl, pr, stream) : launch_depthwise_main(pl, pr, stream);
    if (!st) st = launch_post(pl, ws, dw, stream);
    return st;
}

// The prepared launch (tensor maps and kernel parameters) of a plan on these
// buffers, from the cache or built and cached.
int prepared_for(const wg::Plan& pl, const std::string& pkey, const void* x, const void* dy, void* dw, void* workspace,
                 Prepared* pr)
{
    const void* ws_used = pl.ws_bytes > 0 ? workspace : nullptr;
    const std::string key = prep_key(pkey, x, dy, dw, ws_used);
    {
        std::lock_guard<std::mutex> lk(g_prep_mu);
        auto it = prep_cache().find(key);
        if (it != prep_cache().end()) {
            *pr = it->second;
            return WG_OK;
        }
    }
    const int st = pl.kind == wg::KIND_IGEMM ? prepare_igemm(pl, x, dy, dw, workspace, pr)
                                             : prepare_depthwise(pl, x, dy, dw, workspace, pr);
    if (st) return st;
    std::lock_guard<std::mutex> lk(g_prep_mu);
    if (prep_cache().size() > 4096) prep_cache().clear();
    prep_cache().emplace(key, *pr);
    return WG_OK;
}

// Device buffers and workspace of a call: present, aligned, large enough.
int check_buffers(const wg::Plan& pl, const void* x, const void* dy, const void* dw, const void* workspace,
                  size_t ws_bytes)
{
    if (!x || !dy || !dw) return set_err(WG_ERR_INVALID_ARGUMENT, "x, dy and dw must be non-NULL device pointers");
    if (!aligned16(x) || !aligned16(dy) || !aligned16(dw))
        return set_err(WG_ERR_MISALIGNED, "x, dy and dw must be 16-byte aligned");
    if (pl.ws_bytes > 0) {
        if (!workspace || ws_bytes < pl.ws_bytes) {
            char buf[160];
            snprintf(buf, sizeof buf, "workspace of %zu bytes needed (got %zu%s)", pl.ws_bytes, ws_bytes,
                     workspace ? "" : ", NULL");
            return set_err(WG_ERR_WORKSPACE, buf);
        }
        if (!aligned16(workspace)) return set_err(WG_ERR_MISALIGNED, "workspace must be 16-byte aligned");
    }
    return WG_OK;
}

}  // namespace

extern "C" {

const char* wg_status_string(int s)
{
    switch (s) {
        case WG_OK: return "WG_OK";
        case WG_ERR_INVALID_ARGUMENT: return "WG_ERR_INVALID_ARGUMENT";
        case WG_ERR_NOT_SUPPORTED: return "WG_ERR_NOT_SUPPORTED";
        case WG_ERR_MISALIGNED: return "WG_ERR_MISALIGNED";
        case WG_ERR_WORKSPACE: return "WG_ERR_WORKSPACE";
        case WG_ERR_CUDA: return "WG_ERR_CUDA";
        case WG_ERR_DEVICE_TIMEOUT: return "WG_ERR_DEVICE_TIMEOUT";
        default: return "WG_ERR_UNKNOWN";
    }
}

const char* wg_last_error(void) { return g_err.c_str(); }

int wg_set_mark_event(void* event)
{
    g_mark = static_cast<cudaEvent_t>(event);
    return WG_OK;
}

int wg_problem_normalize(wg_problem* p)
{
    wg::Problem pb;
    std::string err;
    const int st = wg::normalize(p, &pb, &err);
    if (st) return set_err(st, err);
    for (int i = 0; i < p->ndim; ++i) p->out[i] = pb.out[3 - p->ndim + i];
    return WG_OK;
}

int wg_workspace_size(const wg_problem* p, const wg_options* opt, size_t* bytes)
{
    if (!bytes) return set_err(WG_ERR_INVALID_ARGUMENT, "bytes is NULL");
    wg::Plan pl;
    const int st = plan_for(p, opt, &pl);
    if (st) return st;
    *bytes = pl.ws_bytes;
    return WG_OK;
}

int wg_plan_string(const wg_problem* p, const wg_options* opt, char* buf, size_t n)
{
    if (!buf || n == 0) return set_err(WG_ERR_INVALID_ARGUMENT, "buffer is NULL or empty");
    wg::Plan pl;
    const int st = plan_for(p, opt, &pl);
    if (st) return st;
    snprintf(buf, n, "%s", wg::plan_string(pl).c_str());
    return WG_OK;
}

int wg_conv_bwd_weight(const wg_problem* p, const void* x, const void* dy, void* dw, const wg_options* opt,
                       void* workspace, size_t ws_bytes, void* stream)
{
    wg::Plan pl;
    std::string pkey;
    int st = plan_for(p, opt, &pl, &pkey);
    if (st) return st;
    if ((st = check_buffers(pl, x, dy, dw, workspace, ws_bytes))) return st;
    Prepared pr;
    if ((st = prepared_for(pl, pkey, x, dy, dw, workspace, &pr))) return st;
    return launch_call(pl, pr, dw, workspace, static_cast<cudaStream_t>(stream));
}

int wg_conv_bwd_weight_host(const wg_problem* p, const void* x_host, const void* dy_host, void* dw_host,
                            void* x_dev, void* dy_dev, void* dw_dev, const wg_options* opt, void* workspace,
                            size_t ws_bytes, void* stream)
{
    wg::Plan pl;
    std::string pkey;
    int st = plan_for(p, opt, &pl, &pkey);
    if (st) return st;
    if (!x_host || !dy_host || !dw_host)
        return set_err(WG_ERR_INVALID_ARGUMENT, "x_host, dy_host and dw_host must be non-NULL");
    if ((st = check_buffers(pl, x_dev, dy_dev, dw_dev, workspace, ws_bytes))) return st;
    Prepared pr;
    if ((st = prepared_for(pl, pkey, x_dev, dy_dev, dw_dev, workspace, &pr))) return st;
    const wg::Problem& pb = pl.pb;
    const size_t dw_bytes = (size_t)pb.dw_elems * (pb.out_dtype == WG_FP32 ? 4 : 2);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if ((e = cudaMemcpyAsync(x_dev, x_host, (size_t)pb.x_elems * 2, cudaMemcpyHostToDevice, s)) != cudaSuccess)
        return cuda_fail("cudaMemcpyAsync(X)", e);
    if ((e = cudaMemcpyAsync(dy_dev, dy_host, (size_t)pb.dy_elems * 2, cudaMemcpyHostToDevice, s)) != cudaSuccess)
        return cuda_fail("cudaMemcpyAsync(dY)", e);
    if ((st = launch_call(pl, pr, dw_dev, workspace, s))) return st;
    if ((e = cudaMemcpyAsync(dw_host, dw_dev, dw_bytes, cudaMemcpyDeviceToHost, s)) != cudaSuccess)
        return cuda_fail("cudaMemcpyAsync(dW)", e);
    return WG_OK;
}

int wg_selftest_timeout(void* stream)
{
    wg::selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>();
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail("selftest_timeout_kernel launch", e);
    return WG_OK;
}

int wg_check_status(void* stream)
{
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail("cudaStreamSynchronize", e);
    unsigned int v = 0;
    e = cudaMemcpyFromSymbol(&v, wg::g_status, sizeof v);
    if (e != cudaSuccess) return cuda_fail("cudaMemcpyFromSymbol(status)", e);
    if (v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(wg::g_status, &zero, sizeof zero);
        if (e != cudaSuccess) return cuda_fail("cudaMemcpyToSymbol(status)", e);
        return set_err(WG_ERR_DEVICE_TIMEOUT, (v & wg::kStatusBadPlan)
                                                  ? "internal error: a kernel instance got a plan it is not built for"
                                                  : "a kernel's bounded wait ran out");
    }
    return WG_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Entry point for callers that cannot allocate device memory.
//
// wg_conv_bwd_weight takes its split-K workspace from the caller.  Some callers
// cannot provide one: a plug-in whose host application owns every device
// allocation through its own allocator, code running under a fixed device
// memory budget, or a latency-critical path where cudaMalloc's implicit
// synchronisation is not acceptable.  For them the workspace comes from the
// file-scope array below, which every GPU that loads this library holds until
// the process exits.
namespace {

constexpr size_t kNoAllocScratchBytes = 16u << 20;  // 16 MiB per device
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached for the life of the
// process: a cudaDeviceReset ends the context the address belongs to, and the
// cached value must not be used after it.
int noalloc_scratch(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail("cudaGetDevice", e);
    if (dev < 0 || dev >= kMaxDevices) return set_err(WG_ERR_NOT_SUPPORTED, "device ordinal above 63");
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_fail("cudaGetSymbolAddress(scratch)", e);
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return WG_OK;
}

}  // namespace

extern "C" {

int wg_conv_bwd_weight_noalloc(const wg_problem* p, const void* x, const void* dy, void* dw, const wg_options* opt,
                               void* stream)
{
    void* scratch = nullptr;
    int st = noalloc_scratch(&scratch);
    if (st) return st;
    wg_options o{0, WG_MODE_AUTO, 0, 0, WG_KERNEL_AUTO};
    if (opt) o = *opt;
    size_t need = 0;
    st = wg_workspace_size(p, &o, &need);
    if (st) return st;
    if (need > kNoAllocScratchBytes) {
        if (o.split_k != 0) {
            char buf[256];
            snprintf(buf, sizeof buf,
                     "the no-allocation entry point has %zu bytes of scratch; this problem and split degree need %zu",
                     kNoAllocScratchBytes, need);
            return set_err(WG_ERR_WORKSPACE, buf);
        }
        // Automatic split degree: the largest that fits the scratch array.  One
        // partial sum per cluster of Q splits reaches the workspace, so Q * fit
        // splits fit; when not even two partials fit, one split (direct mode,
        // no workspace).  (An automatic mode whose atomic path needs an fp32
        // copy of a 16-bit dW larger than the array takes the two-stage path.)
        if (o.mode == WG_MODE_AUTO) o.mode = WG_MODE_DETERMINISTIC;
        wg::Plan pl1;
        wg_options o1 = o;
        o1.split_k = 1;
        o1.mode = WG_MODE_DETERMINISTIC;
        o1.cluster = 1;
        if ((st = plan_for(p, &o1, &pl1))) return st;
        const size_t per_partial = (size_t)pl1.ws_rows * pl1.ws_nj * pl1.ws_W * 4;
        const size_t fit = kNoAllocScratchBytes / per_partial;
        const int Q = o.cluster > 1 ? o.cluster : 1;
        if (fit < 2) {
            o.split_k = Q;
            if (Q > 1) o.mode = WG_MODE_DIRECT;  // one cluster: its sum is dW
        } else {
            o.split_k = (int)std::min<size_t>(fit * Q, (size_t)(65535 / Q) * Q);
        }
        if ((st = wg_workspace_size(p, &o, &need))) return st;
        if (need > kNoAllocScratchBytes) return set_err(WG_ERR_WORKSPACE, "split-K workspace does not fit the scratch array");
    }
    return wg_conv_bwd_weight(p, x, dy, dw, &o, need ? scratch : nullptr, need ? kNoAllocScratchBytes : 0, stream);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Backward-data (dgrad).
namespace {

struct DgPrepared {
    CUtensorMap tmy, tmw;
    wg::DgParams prm;
};

int dgrad_plan_for(const wg_problem* p, wg::DgPlan* pl, std::string* key_out)
{
    static std::mutex mu;
    static std::map<std::string, wg::DgPlan> cache;
    const wg::DeviceCaps caps = device_caps();
    std::string key;
    if (p) {
        key.assign(reinterpret_cast<const char*>(p), sizeof *p);
        key.append(reinterpret_cast<const char*>(&caps), sizeof caps);
        std::lock_guard<std::mutex> lk(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            *pl = it->second;
            *key_out = key;
            return WG_OK;
        }
    }
    std::string err;
    const int st = wg::make_dgrad_plan(p, caps, pl, &err);
    if (st) return set_err(st, err);
    std::lock_guard<std::mutex> lk(mu);
    if (cache.size() > 1024) cache.clear();
    cache.emplace(key, *pl);
    *key_out = key;
    return WG_OK;
}

int prepare_dgrad(const wg::DgPlan& d, const void* dy, const void* w, void* dx, void* wexp, DgPrepared* out)
{
    const wg::Problem& pb = d.pb;
    {
        const cuuint64_t dims[5] = {(cuuint64_t)pb.G * pb.K, (cuuint64_t)pb.out[2], (cuuint64_t)pb.out[1],
                                    (cuuint64_t)pb.out[0], (cuuint64_t)pb.N};
        const cuuint32_t box[5] = {64, (cuuint32_t)d.PW, (cuuint32_t)d.PH, 1, 1};
        const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        const int st = encode(&out->tmy, pb.in_dtype, const_cast<void*>(dy), dims, box, estr, CU_TENSOR_MAP_SWIZZLE_128B,
                              "dY");
        if (st) return st;
    }
    {
        // W (or its block-diagonal fold) viewed as (C, taps, K, G): k beyond the
        // group's K is out of bounds and reads zero.
        const cuuint64_t dims[5] = {(cuuint64_t)d.Cm, (cuuint64_t)pb.T, (cuuint64_t)d.Km, (cuuint64_t)d.Gb, 1};
        const cuuint32_t box[5] = {64, 1, 64, 1, 1};
        const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
        const int st = encode(&out->tmw, pb.in_dtype, d.Gm > 1 ? wexp : const_cast<void*>(w), dims, box, estr,
                              CU_TENSOR_MAP_SWIZZLE_128B, "W");
        if (st) return st;
    }
    wg::DgParams& q = out->prm;
    memset(&q, 0, sizeof q);
    q.G = d.Gb, q.C = d.Cm, q.K = d.Km;
    q.ch_pix = pb.G * pb.C, q.ch_lim = pb.G * pb.C;
    q.X = pb.filt[2], q.Y = pb.filt[1];
    q.Wi = pb.in[2], q.Hi = pb.in[1], q.Di = pb.in[0];
    q.bw = d.bw, q.bh = d.bh, q.PW = d.PW, q.PH = d.PH;
    q.Nt = d.Nt, q.n_catoms = d.n_catoms, q.n_kc = d.n_kc, q.TG = d.TG;
    q.n_tw = d.n_tw, q.n_th = d.n_th, q.n_td = d.n_td, q.N = pb.N, q.n_ctiles = d.n_ctiles;
    q.n_all = (int)d.n_all;
    q.T = (int)pb.T, q.w_resident = d.w_resident, q.w_bytes = d.w_bytes;
    q.patch_bytes = d.patch_bytes, q.stage_bytes = d.stage_bytes, q.stages = d.stages, q.tmem_cols = d.tmem_cols;
    for (int j = 0; j < 3; ++j) q.dim[j] = d.dim[j];
    q.idesc = wg::make_idesc_f16(pb.in_dtype == WG_BF16, false, true, 128, d.Nt);
    q.out_dtype = pb.out_dtype;
    q.out = dx;
    return WG_OK;
}

std::mutex g_dg_mu;
std::map<std::string, DgPrepared>& dg_cache()
{
    static std::map<std::string, DgPrepared> m;
    return m;
}

}  // namespace

extern "C" {

int wg_bwd_data_plan_string(const wg_problem* p, char* buf, size_t n)
{
    if (!buf || n == 0) return set_err(WG_ERR_INVALID_ARGUMENT, "buffer is NULL or empty");
    wg::DgPlan d;
    std::string key;
    const int st = dgrad_plan_for(p, &d, &key);
    if (st) return st;
    snprintf(buf, n, "%s", wg::dgrad_plan_string(d).c_str());
    return WG_OK;
}

int wg_bwd_data_workspace_size(const wg_problem* p, size_t* bytes)
{
    if (!bytes) return set_err(WG_ERR_INVALID_ARGUMENT, "bytes is NULL");
    wg::DgPlan d;
    std::string key;
    const int st = dgrad_plan_for(p, &d, &key);
    if (st) return st;
    *bytes = d.ws_bytes;
    return WG_OK;
}

int wg_conv_bwd_data(const wg_problem* p, const void* dy, const void* w, void* dx, void* workspace, size_t ws_bytes,
                     void* stream)
{
    wg::DgPlan d;
    std::string pkey;
    int st = dgrad_plan_for(p, &d, &pkey);
    if (st) return st;
    if (!dy || !w || !dx) return set_err(WG_ERR_INVALID_ARGUMENT, "dy, w and dx must be non-NULL device pointers");
    if (!aligned16(dy) || !aligned16(w) || !aligned16(dx))
        return set_err(WG_ERR_MISALIGNED, "dy, w and dx must be 16-byte aligned");
    if (d.ws_bytes > 0) {
        if (!workspace || ws_bytes < d.ws_bytes) {
            char buf[160];
            snprintf(buf, sizeof buf, "workspace of %zu bytes needed (got %zu%s)", d.ws_bytes, ws_bytes,
                     workspace ? "" : ", NULL");
            return set_err(WG_ERR_WORKSPACE, buf);
        }
        if (!aligned16(workspace)) return set_err(WG_ERR_MISALIGNED, "workspace must be 16-byte aligned");
    }
    void* wexp = d.ws_bytes > 0 ? workspace : nullptr;
    const std::string key = prep_key(pkey, dy, w, dx, wexp);
    DgPrepared pr;
    bool hit = false;
    {
        std::lock_guard<std::mutex> lk(g_dg_mu);
        auto it = dg_cache().find(key);
        if (it != dg_cache().end()) pr = it->second, hit = true;
    }
    if (!hit) {
        st = prepare_dgrad(d, dy, w, dx, wexp, &pr);
        if (st) return st;
        std::lock_guard<std::mutex> lk(g_dg_mu);
        if (dg_cache().size() > 4096) dg_cache().clear();
        dg_cache().emplace(key, pr);
    }
    st = ensure_smem(wg::dgrad_kernel, d.smem_bytes);
    if (st) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (d.Gm > 1) {
        const wg::Problem& pb = d.pb;
        const long long n = (long long)d.Gb * d.Km * pb.T * d.Cm;
        const unsigned blocks = (unsigned)std::min<long long>((n + 255) / 256, 4096);
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        unsigned na = 0;
        pdl_config(&cfg, attr, &na, s);
        cfg.gridDim = dim3(blocks);
        cfg.blockDim = dim3(256);
        e = cudaLaunchKernelEx(&cfg, wg::dgrad_fold_w_kernel, static_cast<const uint16_t*>(w),
                               static_cast<uint16_t*>(wexp), pb.G, pb.K, pb.C, (int)pb.T, d.Gm, n);
        if (e != cudaSuccess) return cuda_fail("dgrad_fold_w_kernel launch", e);
    }
    {
        // Like the weight-gradient kernels, a programmatic dependent of the
        // kernel before it (see launch_pre).
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        unsigned na = 0;
        pdl_config(&cfg, attr, &na, s);
        cfg.gridDim = dim3(d.grid[0], d.grid[1], d.grid[2]);
        cfg.blockDim = dim3(d.block);
        cfg.dynamicSmemBytes = (size_t)d.smem_bytes;
        e = cudaLaunchKernelEx(&cfg, wg::dgrad_kernel, pr.tmy, pr.tmw, pr.prm);
        if (e != cudaSuccess) return cuda_fail("dgrad_kernel launch", e);
    }
    if (g_mark && (e = cudaEventRecord(g_mark, s)) != cudaSuccess) return cuda_fail("cudaEventRecord(mark)", e);
    return WG_OK;
}

}  // extern "C"
