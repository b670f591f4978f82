// Host side of the C ABI: argument validation, output shape, the per-shape
// kernel chooser, the plan cache and the launches.
//
// The checks follow the integration concerns listed in "GPU-Accelerating
// MSCRED with CUDA, im2col, GEMM, and a Custom PyTorch Extension" (section
// "Integrating the CUDA Implementation with PyTorch": tensor dimensions,
// device placement, data types, contiguity, error handling): every one of
// them is decided here, before anything is launched, and reported as a
// status code.  The chooser is the per-shape counterpart of the page's
// tile/thread-block tuning (sections "Global Memory and Shared Memory" and
// "Engineering Challenges", kernel configuration).

#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <map>
#include <mutex>
#include <new>
#include <string>
#include <tuple>

#include "internal.h"

using namespace conv2d;

struct conv2d_desc {
    Shape s;
    conv2d_algo_t algo = CONV2D_ALGO_AUTO;
};

namespace {

constexpr int64_t kMaxElems = (int64_t)1 << 40;

int elt_size(conv2d_dtype_t d) { return d == CONV2D_F32 ? 4 : 2; }

int64_t out_extent(int64_t in, int64_t k, int64_t st, int64_t pad, int64_t dil) {
    const int64_t span = in + 2 * pad - dil * (k - 1) - 1;
    return span < 0 ? 0 : span / st + 1;
}

conv2d_status_t make_shape(Shape *s, int N, int C, int H, int W, int K, int R, int S, int stride,
                           int pad, int dil, conv2d_dtype_t dtype, conv2d_layout_t layout) {
    if (N < 1 || C < 1 || H < 1 || W < 1 || K < 1 || R < 1 || S < 1 || stride < 1 || dil < 1 ||
        pad < 0)
        return CONV2D_ERR_INVALID_ARG;
    if (dtype != CONV2D_F32 && dtype != CONV2D_F16 && dtype != CONV2D_BF16)
        return CONV2D_ERR_INVALID_ARG;
    if (layout != CONV2D_NCHW && layout != CONV2D_NHWC) return CONV2D_ERR_INVALID_ARG;
    const int64_t P = out_extent(H, R, stride, pad, dil);
    const int64_t Q = out_extent(W, S, stride, pad, dil);
    if (P < 1 || Q < 1 || P > INT32_MAX || Q > INT32_MAX) return CONV2D_ERR_INVALID_ARG;
    const int64_t xe = (int64_t)N * C * H * W, we = (int64_t)K * C * R * S,
                  ye = (int64_t)N * K * P * Q;
    if (xe >= kMaxElems || we >= kMaxElems || ye >= kMaxElems) return CONV2D_ERR_INVALID_ARG;
    s->N = N; s->C = C; s->H = H; s->W = W; s->K = K; s->R = R; s->S = S;
    s->stride = stride; s->pad = pad; s->dil = dil;
    s->P = (int)P; s->Q = (int)Q;
    s->dtype = dtype; s->layout = layout;
    s->M = (int64_t)N * P * Q;
    s->Kg = (int64_t)C * R * S;
    s->elt = elt_size(dtype);
    return CONV2D_OK;
}

// ------------------------------------------------------------ device info

struct DevInfo {
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    size_t smem_optin = 0;
};

std::mutex g_dev_mu;
std::map<int, DevInfo> g_dev;

conv2d_status_t device_info(int *dev_out, DevInfo *info) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CONV2D_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    auto it = g_dev.find(dev);
    if (it == g_dev.end()) {
        DevInfo d;
        int v = 0;
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return CONV2D_ERR_CUDA;
        d.smem_optin = (size_t)v;
        it = g_dev.emplace(dev, d).first;
    }
    *dev_out = dev;
    *info = it->second;
    return CONV2D_OK;
}

// ------------------------------------------------------------ chooser

// ------------------------------------------------------------ overrides
//
// Switches for tests and A/B measurements (force a kernel, a tile, a grid
// cap, the stall test hook).  They are process-wide, seeded once from the
// environment (CONV2D_<NAME>, e.g. CONV2D_TC_BN=128) the first time the
// library needs them, and changed only through conv2d_set_override.  The
// per-call path reads them as relaxed atomic loads; the plan cache is keyed
// on a generation number that every change bumps, so a plan made under other
// overrides is never reused.

const char *const kOverrideEnv[CONV2D_OVR_COUNT] = {
    "CONV2D_DIRECT",   "CONV2D_CC_TILE",   "CONV2D_CC_SPLIT",  "CONV2D_TC_BN",
    "CONV2D_TC_KSUB",  "CONV2D_TC_IM2COL", "CONV2D_TC_WINDOW", "CONV2D_TC_WINVAR",
    "CONV2D_TC_ROTATE", "CONV2D_TF_VAR",   "CONV2D_FP32_TC",   "CONV2D_DECONV_TC",
    "CONV2D_GRID_CAP", "CONV2D_TEST_WITHHOLD", "CONV2D_TEST_WAIT_KCYCLES", "CONV2D_TC_CTA2"};

std::atomic<int> g_ovr[CONV2D_OVR_COUNT];
std::atomic<int> g_ovr_gen{0};
std::once_flag g_ovr_once;

void seed_overrides() {
    std::call_once(g_ovr_once, [] {
        for (int i = 0; i < CONV2D_OVR_COUNT; ++i) {
            const char *e = std::getenv(kOverrideEnv[i]);
            g_ovr[i].store(e ? std::atoi(e) : -1, std::memory_order_relaxed);
        }
    });
}

}  // namespace

int conv2d::ovr(conv2d_override_t k) {
    seed_overrides();
    return g_ovr[k].load(std::memory_order_relaxed);
}

namespace {

// Estimated time (arbitrary units) of a CUDA-core tile on this layer.
// Each tile has a whole-GPU FFMA rate, measured on GB300 with enough CTAs
// resident (`full_ctas` per SM); with fewer CTAs per SM the rate falls in
// proportion.  Padding of M, K and the reduction to whole tiles is work too.
// Split-K multiplies the CTAs by `split` (each reduces 1/split of the k-tiles)
// at the price of a cluster-wide reduction of the partial tiles.
double cc_cost(const Shape &s, const CudaCoreTile &t, int split, int sms) {
    struct Rate {
        double tflops, full_ctas;
    };
    static const Rate kRates[] = {{30, 3}, {30, 1.5}, {27, 2}, {23, 3},
                                  {22, 3}, {20, 6},   {32, 1.5}, {32, 3}};
    const Rate r = kRates[t.id];
    const int64_t tiles = ((s.M + t.BM - 1) / t.BM) * ((s.K + t.BN - 1) / t.BN);
    const int64_t kt = (s.Kg + t.BK - 1) / t.BK;
    if (split > 1 && kt < 8 * split) return 1e300;         // too little reduction to split
    const double work = (double)tiles * t.BM * t.BN * kt * t.BK;   // FMAs incl. padding
    const double per_sm = (double)tiles * split / sms;
    const double fill = std::min(1.0, per_sm / r.full_ctas);
    // Each cluster rank pays the tap-table build, two cluster barriers and
    // the partial-tile exchange: about as much as 6 k-tiles of its own loop
    // (measured on the MSCRED encoder layers).
    const double reduce = split > 1 ? 1.0 + 6.0 * split / kt : 1.0;
    return work * reduce / (r.tflops * fill);
}

// Direct kernel (short reductions): FFMAs of whole pixel blocks (8 x 32) x
// 32-channel blocks at an effective 30 TFLOP/s, plus about 3 us of launch
// and staging.  In the units of cc_cost(), whose tile rates overestimate
// short reductions by a similar factor: on the MSCRED layer-1 shape on GB300
// the direct kernel measures 24.5 us against 32 us for the best tile.
double dc_cost(const Shape &s) {
    int rows, cols, threads, kc;
    dc_block(&rows, &cols, &threads, &kc);
    const double blocks = (double)s.N * ((s.P + rows - 1) / rows) * ((s.Q + cols - 1) / cols);
    const double fma = blocks * rows * cols * (double)((s.K + kc - 1) / kc * kc) * (double)s.Kg;
    return (2.0 * fma / 30e3 + 3000.0) / 2e-3;
}

conv2d_status_t choose_cc(const Shape &s, const DevInfo &d, Plan *p) {
    const int force_direct = ovr(CONV2D_OVR_DIRECT);
    if (force_direct != 0 && dc_shape_ok(s) && dc_smem_bytes(s) <= d.smem_optin &&
        ovr(CONV2D_OVR_CC_TILE) < 0 && ovr(CONV2D_OVR_CC_SPLIT) < 0) {
        // take the direct kernel when forced, or when it beats every tile
        bool take = force_direct == 1;
        if (!take) {
            take = true;
            const double dc = dc_cost(s);
            for (int id = 0; id < cc_num_tiles() && take; ++id) {
                if (!cc_tile_available(id, s.dtype, 1)) continue;
                const CudaCoreTile t = cc_tile(id);
                if (cc_smem_bytes(s, t) > d.smem_optin) continue;
                if (cc_cost(s, t, 1, d.sm_count) < dc) take = false;
            }
        }
        if (take) {
            p->algo = Algo::Direct;
            p->cc = cc_tile(0);
            p->cc.split = 1;
            p->smem_bytes = dc_smem_bytes(s);
            p->grid = dc_grid(s);
            p->sm_count = d.sm_count;
            return CONV2D_OK;
        }
    }
    if (!cc_shape_ok(s)) return CONV2D_ERR_UNSUPPORTED;
    const int forced = ovr(CONV2D_OVR_CC_TILE);
    const int forced_split = ovr(CONV2D_OVR_CC_SPLIT);
    double best = 1e300;
    int best_id = -1, best_split = 1;
    for (int id = 0; id < cc_num_tiles(); ++id) {
        for (int split : {1, 2, 4}) {
            if (!cc_tile_available(id, s.dtype, split)) continue;
            if (forced >= 0 && id != forced) continue;
            if (forced_split > 0 && split != forced_split) continue;
            const CudaCoreTile t = cc_tile(id);
            const size_t smem = cc_smem_bytes(s, t);
            if (smem > d.smem_optin) continue;
            double c = cc_cost(s, t, split, d.sm_count);
            if (c >= 1e300 && forced_split > 0) c = 1e299;   // a forced split skips the gate
            if (c < best) { best = c; best_id = id; best_split = split; }
        }
    }
    if (best_id < 0) return CONV2D_ERR_UNSUPPORTED;
    p->algo = Algo::CudaCore;
    p->cc = cc_tile(best_id);
    p->cc.split = best_split;
    p->smem_bytes = cc_smem_bytes(s, p->cc);
    p->grid = (int)(((s.M + p->cc.BM - 1) / p->cc.BM) * ((s.K + p->cc.BN - 1) / p->cc.BN)) * best_split;
    p->sm_count = d.sm_count;
    return CONV2D_OK;
}

// Tensor-core plan: BM = 128 output pixels, BN output channels from
// {64, 128, 256}, KSUB 64-channel k-blocks per pipeline stage, and the A mode
// (im2col / plain matrix for 1x1, or padded-row windows for stride-1
// layers).  Measured on GB300, a pipeline stage costs about 0.18 us plus
// 0.09 us per TMA instruction in it, largely independent of the bytes moved
// (TMA fills shared memory at up to about 150 KB/us per SM); the MMAs of one
// k-block take 2 x BN SM cycles.  A tile takes the larger of its MMA time and
// its load time; the layer takes (tiles / SMs rounded up) tiles per SM.  The
// chooser minimises that.
double stage_ns(int instructions, double bytes) {
    return std::max(180.0 + 90.0 * instructions, bytes / 150.0);
}

conv2d_status_t choose_tc(const Shape &s, const DevInfo &d, Plan *p) {
    if (!(d.cc_major == 10 && d.cc_minor == 3)) return CONV2D_ERR_UNSUPPORTED;
    const int64_t cb = (s.C + 63) / 64;
    const int64_t rs = (int64_t)s.R * s.S;
    const int64_t kb = rs * cb;
    const int force_bn = ovr(CONV2D_OVR_TC_BN), force_ks = ovr(CONV2D_OVR_TC_KSUB);
    const int force_win = ovr(CONV2D_OVR_TC_WINDOW);
    const int force_wv = ovr(CONV2D_OVR_TC_WINVAR);
    const bool win_ok = tc_window_ok(s);
    const int wp = s.W + 2 * s.pad;
    const int tr = wp > 0 ? 128 / wp : 0;
    const bool plain = s.R * s.S == 1 && s.stride == 1 && s.pad == 0 && s.C % 64 == 0;
    struct Cand {
        int bn, ks, win_variant;
        double cost;
    };
    Cand best{0, 0, -1, 1e300};
    auto rounds_for = [&](int64_t m_tiles, int bn) {
        const int64_t n_tiles = (s.K + bn - 1) / bn;
        return (m_tiles * n_tiles + d.sm_count - 1) / d.sm_count;
    };
    auto wasteful = [&](int bn) {
        const int64_t n_tiles = (s.K + bn - 1) / bn;
        return force_bn <= 0 && force_wv < 0 && bn > 64 && n_tiles * bn >= s.K + bn / 2 + 1;
    };
    // im2col / plain-matrix variants
    if (force_win != 1) {
        for (int bn : {64, 128, 256}) {
            for (int ks : {1, 2, 3, 4, 6}) {
                if (tc_stages(bn, ks) == 0) continue;
                if (force_bn > 0 && bn != force_bn) continue;
                if (force_ks > 0 && ks != force_ks) continue;
                if (wasteful(bn)) continue;
                const double b_bytes = (double)bn * 128.0;
                double mem;
                if (plain) {
                    mem = ((cb + ks - 1) / ks) * stage_ns(2, ks * (16384.0 + b_bytes));
                } else {
                    const int a_loads = (int)std::min<int64_t>(ks, rs);
                    mem = cb * ((rs + ks - 1) / ks) *
                          stage_ns(a_loads + 1, a_loads * 16384.0 + ks * b_bytes);
                }
                const double mma = kb * 2.0 * bn / 1.9;
                const double cost = (double)rounds_for((s.M + 127) / 128, bn) * std::max(mem, mma);
                if (cost < best.cost) best = Cand{bn, ks, -1, cost};
            }
        }
    }
    // 2-CTA im2col / plain variants (M = 256 over a pair of SMs).  A pair's
    // stage waits for the slower of its two CTAs' loads: measured per-SM
    // ingest is about 0.8x a single CTA's, hence the 1.25 on their load time.
    // Forced on, the best of them wins outright; forced off, none competes.
    const int force_cta2 = ovr(CONV2D_OVR_TC_CTA2);
    if (force_win != 1 && force_cta2 != 0) {
        Cand cb2{0, 0, -1, 1e300};
        for (int bn : {128, 256}) {
            for (int ks : {2, 3, 4}) {
                if (tc_cta2_stages(bn, ks) == 0) continue;
                if (force_bn > 0 && bn != force_bn) continue;
                if (force_ks > 0 && ks != force_ks) continue;
                if (force_cta2 != 1 && wasteful(bn)) continue;
                const double b_bytes = (double)bn * 64.0;   // this CTA's half of the weight tile
                double mem;
                if (plain) {
                    mem = ((cb + ks - 1) / ks) * stage_ns(2, ks * (16384.0 + b_bytes));
                } else {
                    const int a_loads = (int)std::min<int64_t>(ks, rs);
                    mem = cb * ((rs + ks - 1) / ks) *
                          stage_ns(a_loads + 1, a_loads * 16384.0 + ks * b_bytes);
                }
                mem *= 1.25;
                const double mma = kb * 2.0 * bn / 1.9;
                const double cost = (double)rounds_for((s.M + 255) / 256 * 2, bn) * std::max(mem, mma);
                if (cost < cb2.cost) cb2 = Cand{bn, ks, -2, cost};
            }
        }
        if (cb2.bn && (force_cta2 == 1 || cb2.cost < best.cost)) best = cb2;
    }
    // window variants (stride-1 layers)
    if (win_ok && force_win != 0 && force_cta2 != 1) {
        for (int id = 0; id < tc_window_variants(); ++id) {
            if (!tc_window_variant_ok(s, id)) continue;
            if (force_wv >= 0 && id != force_wv) continue;
            const TcWinVariant v = tc_window_variant(id);
            if (force_bn > 0 && v.bn != force_bn) continue;
            if (force_ks > 0 && v.ksub != force_ks && !v.resident) continue;
            if (wasteful(v.bn)) continue;
            const double win_bytes = (double)(tr + (s.R - 1) * s.dil) * wp * 128.0;
            double mem = cb * stage_ns(1, win_bytes);
            if (!v.resident) mem += cb * ((rs + v.ksub - 1) / v.ksub) * stage_ns(1, v.ksub * v.bn * 128.0);
            // few stages in flight: loads are latency-bound unless the weights stay
            // resident; a third stage hides part of that (measured 2-5 % on the
            // 3x3 and 5x5 sweep layers)
            if (!v.resident) mem *= v.stages >= 3 ? 1.15 : 1.25;
            const double mma = kb * 2.0 * v.bn / 1.9;
            const double cost = (double)rounds_for((int64_t)s.N * ((s.P + tr - 1) / tr), v.bn) *
                                std::max(mem, mma);
            if (cost < best.cost) best = Cand{v.bn, v.ksub, id, cost};
        }
    }
    if (best.bn == 0) return CONV2D_ERR_UNSUPPORTED;
    TcTile t;
    t.BN = best.bn;
    t.ksub = best.ks;
    t.cta2 = best.win_variant == -2;
    t.window = best.win_variant >= 0;
    t.win_variant = t.window ? best.win_variant : -1;
    t.stages = t.window ? tc_window_variant(best.win_variant).stages
               : t.cta2 ? tc_cta2_stages(best.bn, best.ks) : tc_stages(best.bn, best.ks);
    t.tma_store = true;
    t.force_im2col = ovr(CONV2D_OVR_TC_IM2COL) == 1;
    t.rotate = ovr(CONV2D_OVR_TC_ROTATE) != 0;
    p->algo = Algo::TensorCore;
    p->tc = t;
    p->smem_bytes = t.window ? tc_window_smem_bytes(t) : tc_smem_bytes(t);
    if (p->smem_bytes > d.smem_optin) return CONV2D_ERR_UNSUPPORTED;
    const int64_t m_tiles = t.window ? (int64_t)s.N * ((s.P + tr - 1) / tr) : (s.M + 127) / 128;
    const int64_t tiles = m_tiles * ((s.K + best.bn - 1) / best.bn);
    p->grid = (int)std::min<int64_t>(tiles, d.sm_count);
    if (ovr(CONV2D_OVR_GRID_CAP) > 0) p->grid = std::min(p->grid, ovr(CONV2D_OVR_GRID_CAP));
    if (t.cta2) p->grid = std::max(2, p->grid / 2 * 2);   // whole clusters of two
    p->sm_count = d.sm_count;
    return CONV2D_OK;
}

// fp32 split-precision tensor-core plan (3xTF32).  Each variant carries its
// measured time per 32-element stage of one 128 x BN tile; a tile also pays
// about 2 us of pipeline fill and epilogue, a launch about 2 us.  Persistent
// CTAs run ceil(tiles / SMs) tiles each.  Result in nanoseconds, comparable
// with cc_cost() * 2e-3.
double tf_cost_ns(const Shape &s, const TfTile &t, int sms) {
    const int64_t ntn = (s.K + t.BN - 1) / t.BN;
    const int64_t tiles = ((s.M + 127) / 128) * ntn;
    int64_t grid = std::min<int64_t>(tiles, sms);
    if (t.resb) grid = std::max(ntn, grid / ntn * ntn);   // a CTA keeps one output-channel tile
    const int64_t rounds = (tiles + grid - 1) / grid;
    const int64_t kt = (s.Kg + 31) / 32;
    return 2000.0 + (double)rounds * ((double)kt * t.stage_ns + 2000.0);
}

conv2d_status_t choose_tf(const Shape &s, const DevInfo &d, Plan *p, double *cost_ns,
                          bool lstm = false) {
    if (!(d.cc_major == 10 && d.cc_minor == 3) || !tf_shape_ok(s)) return CONV2D_ERR_UNSUPPORTED;
    const int forced = ovr(CONV2D_OVR_TF_VAR);
    double best = 1e300;
    int best_id = -1;
    for (int id = 0; id < tf_num_variants(); ++id) {
        if (forced >= 0 && id != forced) continue;
        const TfTile t = tf_variant(id);
        if (lstm && !tf_lstm_variant(id)) continue;
        if (tf_smem_bytes(s, t) > d.smem_optin) continue;
        // a tile much wider than K wastes tensor-core work
        if (forced < 0 && t.BN > 32 && s.K <= t.BN / 2) continue;
        const double c = tf_cost_ns(s, t, d.sm_count);
        if (c < best) { best = c; best_id = id; }
    }
    if (best_id < 0) return CONV2D_ERR_UNSUPPORTED;
    p->algo = Algo::Tf32x3;
    p->tf = tf_variant(best_id);
    p->smem_bytes = tf_smem_bytes(s, p->tf);
    const int64_t tiles = ((s.M + 127) / 128) * ((s.K + p->tf.BN - 1) / p->tf.BN);
    p->grid = (int)std::min<int64_t>(tiles, d.sm_count);
    if (ovr(CONV2D_OVR_GRID_CAP) > 0) p->grid = std::min(p->grid, ovr(CONV2D_OVR_GRID_CAP));
    p->sm_count = d.sm_count;
    if (cost_ns) *cost_ns = best;
    return CONV2D_OK;
}

bool aligned16(const Tensors &t) {
    auto a = [](const void *p) { return ((uintptr_t)p & 15) == 0; };
    return a(t.x) && a(t.w) && a(t.y) && (t.bias == nullptr || ((uintptr_t)t.bias & 1) == 0);
}

// Plans are cached per (device, shape, dtype, layout, algo, alignment class)
// and the override generation (conv2d_set_override bumps it).
using PlanKey = std::tuple<int, int, int, int, int, int, int, int, int, int, int, int, int, int, int,
                           int>;

std::mutex g_plan_mu;
std::map<PlanKey, Plan> g_plans;

conv2d_status_t get_plan(const Shape &s, conv2d_algo_t algo, const Tensors *t, Plan *out) {
    int dev = 0;
    DevInfo d;
    conv2d_status_t st = device_info(&dev, &d);
    if (st != CONV2D_OK) return st;
    const bool al = t == nullptr || aligned16(*t);
    seed_overrides();
    const PlanKey key{dev, s.N, s.C, s.H, s.W, s.K, s.R, s.S, s.stride, s.pad, s.dil,
                      (int)s.dtype, (int)s.layout, (int)algo, al ? 1 : 0,
                      g_ovr_gen.load(std::memory_order_acquire)};
    {
        std::lock_guard<std::mutex> lk(g_plan_mu);
        auto it = g_plans.find(key);
        if (it != g_plans.end()) { *out = it->second; return CONV2D_OK; }
    }
    Plan p{};
    const bool tc_ok = tc_shape_ok(s, t);
    if (s.dtype == CONV2D_F32) {
        // fp32: FFMA on CUDA cores, or 3xTF32 on tensor cores, whichever the
        // cost models expect to be faster (CONV2D_FP32_TC=0 keeps FFMA).
        if (algo == CONV2D_ALGO_TENSOR_CORE) {
            st = choose_tf(s, d, &p, nullptr);
        } else if (algo == CONV2D_ALGO_CUDA_CORE) {
            st = choose_cc(s, d, &p);
        } else {
            Plan ptf{};
            double tf_ns = 1e300;
            const bool tf_on = ovr(CONV2D_OVR_FP32_TC) != 0 &&
                               choose_tf(s, d, &ptf, &tf_ns) == CONV2D_OK;
            st = choose_cc(s, d, &p);
            const double cc_ns = st != CONV2D_OK ? 1e300
                                 : p.algo == Algo::Direct ? dc_cost(s) * 2e-3
                                 : cc_cost(s, p.cc, p.cc.split, d.sm_count) * 2e-3;
            if (tf_on && (st != CONV2D_OK || tf_ns < cc_ns)) {
                p = ptf;
                st = CONV2D_OK;
            }
        }
    } else if (algo == CONV2D_ALGO_TENSOR_CORE) {
        if (!tc_ok) return CONV2D_ERR_UNSUPPORTED;
        st = choose_tc(s, d, &p);
    } else if (algo == CONV2D_ALGO_CUDA_CORE) {
        st = choose_cc(s, d, &p);
    } else {
        st = tc_ok ? choose_tc(s, d, &p) : CONV2D_ERR_UNSUPPORTED;
        if (st != CONV2D_OK) st = choose_cc(s, d, &p);
    }
    if (st != CONV2D_OK) return st;
    if (std::getenv("CONV2D_LOG")) {
        if (p.algo == Algo::TensorCore)
            std::fprintf(stderr, "[conv2d] tensor-core BM=128 BN=%d ksub=%d stages=%d grid=%d smem=%zu\n",
                         p.tc.BN, p.tc.ksub, p.tc.stages, p.grid, p.smem_bytes);
        else if (p.algo == Algo::Tf32x3)
            std::fprintf(stderr, "[conv2d] tensor-core 3xtf32 BM=128 BN=%d stages=%d producers=%d grid=%d smem=%zu\n",
                         p.tf.BN, p.tf.stages, p.tf.nprod, p.grid, p.smem_bytes);
        else
            std::fprintf(stderr, "[conv2d] cuda-core tile=%d (%dx%dx%d, %dx%d/thread) split=%d grid=%d smem=%zu\n",
                         p.cc.id, p.cc.BM, p.cc.BN, p.cc.BK, p.cc.TM, p.cc.TN, p.cc.split, p.grid, p.smem_bytes);
    }
    std::lock_guard<std::mutex> lk(g_plan_mu);
    g_plans[key] = p;
    *out = p;
    return CONV2D_OK;
}

// ------------------------------------------------------------ pointer checks

// The pointer must be device (or managed) memory of `dev`; returns false for
// host memory, which a kernel could not (or should not) dereference.
bool is_device_ptr(const void *p, int dev) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeDevice) return a.device == dev;
    if (a.type == cudaMemoryTypeManaged) return true;
    return false;
}

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    if (!a || !b) return false;
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + nb && b0 < a0 + na;
}

conv2d_status_t check_tensors(const Shape &s, const Tensors &t, cudaStream_t stream) {
    if (!t.x || !t.w || !t.y) return CONV2D_ERR_INVALID_ARG;
    const uintptr_t mask = (uintptr_t)s.elt - 1;
    if (((uintptr_t)t.x & mask) || ((uintptr_t)t.w & mask) || ((uintptr_t)t.y & mask) ||
        (t.bias && ((uintptr_t)t.bias & mask)))
        return CONV2D_ERR_MISALIGNED;
    const size_t xb = (size_t)s.x_elems() * s.elt, wb = (size_t)s.w_elems() * s.elt,
                 yb = (size_t)s.y_elems() * s.elt, bb = (size_t)s.K * s.elt;
    if (overlaps(t.y, yb, t.x, xb) || overlaps(t.y, yb, t.w, wb) ||
        (t.bias && overlaps(t.y, yb, t.bias, bb)))
        return CONV2D_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CONV2D_ERR_CUDA;
    // cudaStreamGetDevice invalidates an ongoing stream capture, so the
    // stream's device is checked only when the stream is not capturing.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (stream && cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        cudaGetLastError();
        return CONV2D_ERR_INVALID_ARG;
    }
    if (stream && cap == cudaStreamCaptureStatusNone) {
        int sdev = -1;
        if (cudaStreamGetDevice(stream, &sdev) != cudaSuccess) {
            cudaGetLastError();
            return CONV2D_ERR_INVALID_ARG;
        }
        if (sdev != dev) return CONV2D_ERR_INVALID_ARG;
    }
    if (!is_device_ptr(t.x, dev) || !is_device_ptr(t.w, dev) || !is_device_ptr(t.y, dev) ||
        (t.bias && !is_device_ptr(t.bias, dev)))
        return CONV2D_ERR_INVALID_ARG;
    return CONV2D_OK;
}

conv2d_status_t run(const Shape &s, conv2d_algo_t algo, const Tensors &t, cudaStream_t stream) {
    conv2d_status_t st = check_tensors(s, t, stream);
    if (st != CONV2D_OK) return st;
    Plan p;
    st = get_plan(s, algo, &t, &p);
    if (st != CONV2D_OK) return st;
    if (p.algo == Algo::TensorCore) return tc_launch(s, p, t, stream);
    if (p.algo == Algo::Tf32x3) return tf_launch(s, p, t, stream);
    if (p.algo == Algo::Direct) return dc_launch(s, p, t, stream);
    return cc_launch(s, p, t, stream);
}

}  // namespace

extern "C" {

conv2d_status_t conv2d_desc_create(conv2d_desc_t *out, int N, int C, int H, int W, int K, int R,
                                   int S, int stride, int pad, int dil, conv2d_dtype_t dtype,
                                   conv2d_layout_t layout) {
    if (!out) return CONV2D_ERR_INVALID_ARG;
    Shape s;
    conv2d_status_t st = make_shape(&s, N, C, H, W, K, R, S, stride, pad, dil, dtype, layout);
    if (st != CONV2D_OK) return st;
    conv2d_desc *d = new (std::nothrow) conv2d_desc;
    if (!d) return CONV2D_ERR_INTERNAL;
    d->s = s;
    *out = d;
    return CONV2D_OK;
}

conv2d_status_t conv2d_desc_destroy(conv2d_desc_t desc) {
    delete desc;
    return CONV2D_OK;
}

conv2d_status_t conv2d_output_dims(conv2d_desc_t desc, int *P, int *Q) {
    if (!desc || !P || !Q) return CONV2D_ERR_INVALID_ARG;
    *P = desc->s.P;
    *Q = desc->s.Q;
    return CONV2D_OK;
}

conv2d_status_t conv2d_workspace_bytes(conv2d_desc_t desc, size_t *bytes) {
    if (!desc || !bytes) return CONV2D_ERR_INVALID_ARG;
    *bytes = 0;
    return CONV2D_OK;
}

conv2d_status_t conv2d_desc_set_algo(conv2d_desc_t desc, conv2d_algo_t algo) {
    if (!desc) return CONV2D_ERR_INVALID_ARG;
    if (algo != CONV2D_ALGO_AUTO && algo != CONV2D_ALGO_CUDA_CORE && algo != CONV2D_ALGO_TENSOR_CORE)
        return CONV2D_ERR_INVALID_ARG;
    if (algo == CONV2D_ALGO_TENSOR_CORE && !tc_shape_ok(desc->s, nullptr) && !tf_shape_ok(desc->s))
        return CONV2D_ERR_UNSUPPORTED;
    if (algo == CONV2D_ALGO_CUDA_CORE && !cc_shape_ok(desc->s) && !dc_shape_ok(desc->s))
        return CONV2D_ERR_UNSUPPORTED;
    desc->algo = algo;
    return CONV2D_OK;
}

conv2d_status_t conv2d_desc_plan(conv2d_desc_t desc, char *buf, size_t len) {
    if (!desc || !buf || len == 0) return CONV2D_ERR_INVALID_ARG;
    Plan p;
    conv2d_status_t st = get_plan(desc->s, desc->algo, nullptr, &p);
    if (st != CONV2D_OK) return st;
    if (p.algo == Algo::TensorCore)
        std::snprintf(buf, len, "tensor_core tcgen05 BM=128 BN=%d BK=64 ksub=%d stages=%d grid=%d smem=%zu %sa=%s%s",
                      p.tc.BN, p.tc.ksub, p.tc.stages, p.grid, p.smem_bytes, p.tc.cta2 ? "cta2 " : "",
                      p.tc.window && tc_window_variant(p.tc.win_variant).resident ? "resident-w " : "",
                      p.tc.window ? "window"
                      : (desc->s.R == 1 && desc->s.S == 1 && desc->s.stride == 1 && desc->s.pad == 0 &&
                         !p.tc.force_im2col) ? "tile" : "im2col");
    else if (p.algo == Algo::Direct) {
        int rows, cols, threads, kc;
        dc_block(&rows, &cols, &threads, &kc);
        std::snprintf(buf, len, "cuda_core direct ffma block=%dx%dpx kc=%d threads=%d grid=%d smem=%zu",
                      rows, cols, kc, threads, p.grid, p.smem_bytes);
    } else if (p.algo == Algo::Tf32x3)
        std::snprintf(buf, len, "tensor_core tcgen05 3xtf32 BM=128 BN=%d BK=32 stages=%d producers=%d groups=%d%s grid=%d smem=%zu",
                      p.tf.BN, p.tf.stages, p.tf.nprod * 32, p.tf.ngrp, p.tf.resb ? " resident-w" : "", p.grid,
                      p.smem_bytes);
    else
        std::snprintf(buf, len, "cuda_core ffma BM=%d BN=%d BK=%d TM=%d TN=%d threads=%d split=%d grid=%d smem=%zu",
                      p.cc.BM, p.cc.BN, p.cc.BK, p.cc.TM, p.cc.TN, p.cc.threads, p.cc.split, p.grid,
                      p.smem_bytes);
    return CONV2D_OK;
}

conv2d_status_t conv2d_forward_desc(conv2d_desc_t desc, const void *x, const void *w,
                                    const void *bias, void *y, cudaStream_t stream) {
    if (!desc) return CONV2D_ERR_INVALID_ARG;
    return run(desc->s, desc->algo, Tensors{x, w, bias, y}, stream);
}

conv2d_status_t conv2d_forward(const void *x, const void *w, const void *bias, void *y, int N,
                               int C, int H, int W, int K, int R, int S, int stride, int pad,
                               int dil, conv2d_dtype_t dtype, conv2d_layout_t layout,
                               cudaStream_t stream) {
    Shape s;
    conv2d_status_t st = make_shape(&s, N, C, H, W, K, R, S, stride, pad, dil, dtype, layout);
    if (st != CONV2D_OK) return st;
    return run(s, CONV2D_ALGO_AUTO, Tensors{x, w, bias, y}, stream);
}

conv2d_status_t conv2d_deconv_output_dims(int P, int Q, int R, int S, int stride, int pad, int dil,
                                          int out_pad, int *H, int *W) {
    if (!H || !W || P < 1 || Q < 1 || R < 1 || S < 1 || stride < 1 || dil < 1 || pad < 0 ||
        out_pad < 0 || out_pad >= std::max(stride, dil))
        return CONV2D_ERR_INVALID_ARG;
    const int64_t h = (int64_t)(P - 1) * stride - 2 * (int64_t)pad + (int64_t)dil * (R - 1) + 1 + out_pad;
    const int64_t w = (int64_t)(Q - 1) * stride - 2 * (int64_t)pad + (int64_t)dil * (S - 1) + 1 + out_pad;
    if (h < 1 || w < 1 || h > INT32_MAX || w > INT32_MAX) return CONV2D_ERR_INVALID_ARG;
    *H = (int)h;
    *W = (int)w;
    return CONV2D_OK;
}

conv2d_status_t conv2d_deconv_forward(const void *x, const void *w, const void *bias, void *y,
                                      int N, int K, int P, int Q, int C, int R, int S, int stride,
                                      int pad, int dil, int out_pad, conv2d_dtype_t dtype,
                                      conv2d_layout_t layout, cudaStream_t stream) {
    int H = 0, W = 0;
    if (N < 1 || K < 1 || C < 1) return CONV2D_ERR_INVALID_ARG;
    conv2d_status_t st = conv2d_deconv_output_dims(P, Q, R, S, stride, pad, dil, out_pad, &H, &W);
    if (st != CONV2D_OK) return st;
    if (dtype != CONV2D_F32 && dtype != CONV2D_F16 && dtype != CONV2D_BF16) return CONV2D_ERR_INVALID_ARG;
    if (layout != CONV2D_NCHW && layout != CONV2D_NHWC) return CONV2D_ERR_INVALID_ARG;
    if (dtype != CONV2D_F32 || layout != CONV2D_NCHW) return CONV2D_ERR_UNSUPPORTED;
    const int64_t xe = (int64_t)N * K * P * Q, we = (int64_t)K * C * R * S, ye = (int64_t)N * C * H * W;
    if (xe >= kMaxElems || we >= kMaxElems || ye >= kMaxElems) return CONV2D_ERR_INVALID_ARG;
    if (!x || !w || !y) return CONV2D_ERR_INVALID_ARG;
    if (((uintptr_t)x & 3) || ((uintptr_t)w & 3) || ((uintptr_t)y & 3) || (bias && ((uintptr_t)bias & 3)))
        return CONV2D_ERR_MISALIGNED;
    if (overlaps(y, (size_t)ye * 4, x, (size_t)xe * 4) || overlaps(y, (size_t)ye * 4, w, (size_t)we * 4) ||
        (bias && overlaps(y, (size_t)ye * 4, bias, (size_t)C * 4)))
        return CONV2D_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CONV2D_ERR_CUDA;
    if (!is_device_ptr(x, dev) || !is_device_ptr(w, dev) || !is_device_ptr(y, dev) ||
        (bias && !is_device_ptr(bias, dev)))
        return CONV2D_ERR_INVALID_ARG;
    // Tensor cores first: split the outputs into the stride^2 residue classes
    // (h mod stride, w mod stride).  Within a class every output takes the
    // same filter rows r (those with r*dil = h + pad mod stride) and columns,
    // reading input row i + e_r for class row i: a stride-1 gather, run on
    // the 3xTF32 kernel with its outputs written in place into y.  A class
    // without taps (only bias) or a shape the kernel cannot hold uses the
    // gather kernel for the whole layer.  So does a layer with at most 8
    // outputs channels: the tensor-core tile is at least 32 channels wide
    // and its gather of the inputs costs the same however few of them are
    // used, while the gather kernel's work shrinks with its channel block.
    // CONV2D_DECONV_TC=1 / 0 forces either path.
    DevInfo d;
    int dev2 = 0;
    const int force_tc = ovr(CONV2D_OVR_DECONV_TC);
    const bool try_tc = force_tc == 1 || (force_tc < 0 && C > 8);
    if (try_tc && R <= 8 && S <= 8 && device_info(&dev2, &d) == CONV2D_OK &&
        d.cc_major == 10 && d.cc_minor == 3) {
        struct Cls { int a, b; TfDeconv dv; Shape s; Plan p; };
        Cls cls[64];
        int nc = 0;
        bool ok = stride * stride <= 64;
        for (int a = 0; ok && a < stride; ++a) {
            for (int b = 0; ok && b < stride; ++b) {
                const int Pc = a < H ? (H - a + stride - 1) / stride : 0;
                const int Qc = b < W ? (W - b + stride - 1) / stride : 0;
                if (Pc == 0 || Qc == 0) continue;
                TfDeconv dv{};
                dv.H = H; dv.W = W; dv.a = a; dv.b = b; dv.st = stride; dv.R = R; dv.S = S;
                for (int r = 0; r < R; ++r) {
                    const int t = a + pad - r * dil;
                    if (((t % stride) + stride) % stride == 0) {
                        dv.r[dv.J] = r;
                        dv.e[dv.J] = t >= 0 ? t / stride : -((-t) / stride);
                        ++dv.J;
                    }
                }
                for (int q = 0; q < S; ++q) {
                    const int t = b + pad - q * dil;
                    if (((t % stride) + stride) % stride == 0) {
                        dv.s[dv.L] = q;
                        dv.f[dv.L] = t >= 0 ? t / stride : -((-t) / stride);
                        ++dv.L;
                    }
                }
                if (dv.J == 0 || dv.L == 0) { ok = false; break; }
                Shape cs{};
                cs.N = N; cs.C = K; cs.H = P; cs.W = Q; cs.K = C; cs.R = dv.J; cs.S = dv.L;
                cs.stride = 1; cs.pad = 0; cs.dil = 1; cs.P = Pc; cs.Q = Qc;
                cs.dtype = CONV2D_F32; cs.layout = CONV2D_NCHW;
                cs.M = (int64_t)N * Pc * Qc;
                cs.Kg = (int64_t)K * dv.J * dv.L;
                cs.elt = 4;
                Plan pl{};
                if (choose_tf(cs, d, &pl, nullptr) != CONV2D_OK) { ok = false; break; }
                cls[nc++] = Cls{a, b, dv, cs, pl};
            }
        }
        if (ok && nc > 0) {
            for (int i = 0; i < nc; ++i) {
                const conv2d_status_t st2 = tf_launch(cls[i].s, cls[i].p, Tensors{x, w, bias, y}, stream,
                                                      nullptr, &cls[i].dv);
                if (st2 != CONV2D_OK) return st2;
            }
            return CONV2D_OK;
        }
    }
    return dv_launch(static_cast<const float *>(x), static_cast<const float *>(w),
                     static_cast<const float *>(bias), static_cast<float *>(y), N, K, P, Q, C, R, S,
                     H, W, stride, pad, dil, stream);
}

conv2d_status_t conv2d_signature_matrices(const float *series, int n_signals, int T,
                                          const int *windows, int n_windows, int t_first,
                                          int n_steps, float *out, cudaStream_t stream) {
    if (!series || !out || !windows) return CONV2D_ERR_INVALID_ARG;
    if (n_signals < 1 || n_signals > 128 || T < 1 || n_windows < 1 || n_windows > 8 || n_steps < 1)
        return CONV2D_ERR_INVALID_ARG;
    int wmax = 0;
    for (int c = 0; c < n_windows; ++c) {
        if (windows[c] < 1) return CONV2D_ERR_INVALID_ARG;
        wmax = std::max(wmax, windows[c]);
    }
    if (wmax > t_first || (int64_t)t_first + n_steps - 1 > T) return CONV2D_ERR_INVALID_ARG;
    if (((uintptr_t)series & 3) || ((uintptr_t)out & 3)) return CONV2D_ERR_MISALIGNED;
    const size_t sb = (size_t)n_signals * T * sizeof(float);
    const size_t ob = (size_t)n_steps * n_windows * n_signals * n_signals * sizeof(float);
    if (overlaps(out, ob, series, sb)) return CONV2D_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CONV2D_ERR_CUDA;
    if (!is_device_ptr(series, dev) || !is_device_ptr(out, dev)) return CONV2D_ERR_INVALID_ARG;
    return sig_launch(series, n_signals, T, windows, n_windows, t_first, n_steps, out, stream);
}

conv2d_status_t conv2d_convlstm_cell(const float *xh, const float *w, const float *bias,
                                     const float *c_prev, float *c_next, float *h_next,
                                     int N, int Cx, int Ch, int H, int W, int R, int S, int pad,
                                     int dil, long long h_img_stride, cudaStream_t stream) {
    if (Cx < 0 || Ch < 1) return CONV2D_ERR_INVALID_ARG;
    Shape s;
    conv2d_status_t st = make_shape(&s, N, Cx + Ch, H, W, 4 * Ch, R, S, 1, pad, dil, CONV2D_F32,
                                    CONV2D_NCHW);
    if (st != CONV2D_OK) return st;
    if (s.P != H || s.Q != W) return CONV2D_ERR_INVALID_ARG;            // the state keeps H x W
    const int64_t plane = (int64_t)Ch * H * W;
    if (h_img_stride < plane) return CONV2D_ERR_INVALID_ARG;
    if (!xh || !w || !c_prev || !c_next || !h_next) return CONV2D_ERR_INVALID_ARG;
    const uintptr_t m4 = 3;
    if (((uintptr_t)xh & m4) || ((uintptr_t)w & m4) || ((uintptr_t)c_prev & m4) ||
        ((uintptr_t)c_next & m4) || ((uintptr_t)h_next & m4) || (bias && ((uintptr_t)bias & m4)))
        return CONV2D_ERR_MISALIGNED;
    // outputs must not overlap the inputs they are computed from
    const size_t xb = (size_t)s.x_elems() * 4, wb = (size_t)s.w_elems() * 4, cb = (size_t)N * plane * 4;
    const size_t hb = ((size_t)(N - 1) * (size_t)h_img_stride + (size_t)plane) * 4;
    if (overlaps(c_next, cb, xh, xb) || overlaps(c_next, cb, w, wb) || overlaps(c_next, cb, c_prev, cb) ||
        overlaps(h_next, hb, xh, xb) || overlaps(h_next, hb, w, wb) || overlaps(h_next, hb, c_prev, cb) ||
        overlaps(h_next, hb, c_next, cb) ||
        (bias && (overlaps(c_next, cb, bias, (size_t)s.K * 4) || overlaps(h_next, hb, bias, (size_t)s.K * 4))))
        return CONV2D_ERR_INVALID_ARG;
    int dev = 0;
    DevInfo d;
    st = device_info(&dev, &d);
    if (st != CONV2D_OK) return st;
    if (!is_device_ptr(xh, dev) || !is_device_ptr(w, dev) || !is_device_ptr(c_prev, dev) ||
        !is_device_ptr(c_next, dev) || !is_device_ptr(h_next, dev) || (bias && !is_device_ptr(bias, dev)))
        return CONV2D_ERR_INVALID_ARG;
    Plan p{};
    st = choose_tf(s, d, &p, nullptr, true);
    if (st != CONV2D_OK) return st;
    const TfLstm lstm{c_prev, c_next, h_next, (int64_t)h_img_stride};
    return tf_launch(s, p, Tensors{xh, w, bias, nullptr}, stream, &lstm);
}

const char *conv2d_status_string(conv2d_status_t status) {
    switch (status) {
        case CONV2D_OK: return "ok";
        case CONV2D_ERR_INVALID_ARG: return "invalid argument";
        case CONV2D_ERR_UNSUPPORTED: return "unsupported configuration";
        case CONV2D_ERR_MISALIGNED: return "misaligned pointer";
        case CONV2D_ERR_CUDA: return "CUDA error";
        case CONV2D_ERR_TIMEOUT: return "kernel barrier wait timed out";
        case CONV2D_ERR_INTERNAL: return "internal error";
    }
    return "unknown status";
}

conv2d_status_t conv2d_get_device_status(void) { return status_read_and_clear(); }

conv2d_status_t conv2d_set_override(conv2d_override_t key, int value) {
    if ((int)key < 0 || (int)key >= CONV2D_OVR_COUNT) return CONV2D_ERR_INVALID_ARG;
    if (value < -1) return CONV2D_ERR_INVALID_ARG;
    seed_overrides();
    std::lock_guard<std::mutex> lk(g_plan_mu);
    g_ovr[key].store(value, std::memory_order_relaxed);
    g_ovr_gen.fetch_add(1, std::memory_order_acq_rel);
    g_plans.clear();   // plans made under the old value are never looked up again
    return CONV2D_OK;
}

conv2d_status_t conv2d_get_override(conv2d_override_t key, int *value) {
    if ((int)key < 0 || (int)key >= CONV2D_OVR_COUNT || !value) return CONV2D_ERR_INVALID_ARG;
    *value = ovr(key);
    return CONV2D_OK;
}

conv2d_status_t conv2d_variant_count(conv2d_family_t family, int *count) {
    if (!count) return CONV2D_ERR_INVALID_ARG;
    switch (family) {
        case CONV2D_FAMILY_CUDA_CORE_TILE: *count = cc_num_tiles(); return CONV2D_OK;
        case CONV2D_FAMILY_TENSOR_CORE: *count = tc_num_variants(); return CONV2D_OK;
        case CONV2D_FAMILY_TENSOR_CORE_WINDOW: *count = tc_window_variants(); return CONV2D_OK;
        case CONV2D_FAMILY_TF32X3: *count = tf_num_variants(); return CONV2D_OK;
        case CONV2D_FAMILY_TENSOR_CORE_PAIR: *count = tc_cta2_num_variants(); return CONV2D_OK;
    }
    return CONV2D_ERR_INVALID_ARG;
}

int conv2d_version(void) { return 100; }

}  // extern "C"
