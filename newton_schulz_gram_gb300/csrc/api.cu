// C ABI, planner and workspace of the Gram Newton-Schulz library.
//
// The planner turns one bucket of G equal-shaped matrices into a fixed list
// of grouped launches:
//   sum of squares -> scale / cast / transpose (fp16 X and X^T) ->
//   GEMM phases of Dion3 Algorithm 3 (or Algorithm 1 for square matrices).
// Every GEMM phase covers all matrices of the bucket (or of a chunk of it),
// so small matrices still fill the chip; per-tile arithmetic never depends on
// G, so a matrix gives bit-identical results alone or inside a bucket.
//
// fp16 range: the fp16 copy is X~ = 2^k X (k = min(6, floor(log2 n) / 2)) and
// every Gram-state matrix is carried as s = 4^k times its value (R~ = s R,
// Z~ = s Z, RZ~ = s RZ; Q unscaled). The epilogue constants absorb the
// scale exactly (powers of two): Z~ = b R~ + (c/s) R~R~,
// Q' = (1/s) Q Z~ + a Q, RZ~ = (1/s) R~ Z~ + a R~, R~' = (1/s) Z~ RZ~ + a RZ~,
// O = 2^-k Q X~. This keeps the entries of R (about 1/(n sqrt(m)) off the
// diagonal at t = 0) out of the fp16 subnormal range.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "dion3.cuh"
#include "elementwise.cuh"
#include "gemm.cuh"
#include "gns.h"

namespace gns {
namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& msg) {
    g_last_error = msg;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(GNS_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define CK(call)                                                        \
    do {                                                                \
        cudaError_t e_ = static_cast<cudaError_t>(call);                \
        if (e_ != cudaSuccess) return cuda_fail(e_, #call);             \
    } while (0)

#define RET(call)                 \
    do {                          \
        int r_ = (call);          \
        if (r_ != GNS_OK) return r_; \
    } while (0)

constexpr float kQuintic[3] = {3.4445f, -4.7750f, 2.0315f};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
long long round_up_ll(long long v, long long a) { return (v + a - 1) / a * a; }

struct DeviceState {
    int device = -1;
    int num_sms = 0;
    int cc_major = 0, cc_minor = 0;
    char* ws = nullptr;
    size_t ws_bytes = 0;
    int* err = nullptr;      // status block: [0] status word, [1] abort mark (see DevStatus)
    int epoch = 0;           // number of the current call on this device
    DevStatus status{};      // the current call's device-side error reporting
    float* stage = nullptr;  // device staging for the host-buffer entry point
    size_t stage_bytes = 0;
    cudaStream_t h2d = nullptr, d2h = nullptr;  // copy streams of the host-buffer entry point
};

std::mutex g_mu;
std::map<int, DeviceState> g_dev;

int get_state(DeviceState** out) {
    int dev = 0;
    CK(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState& st = g_dev[dev];
    if (st.device < 0) {
        CK(cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev));
        CK(cudaDeviceGetAttribute(&st.cc_major, cudaDevAttrComputeCapabilityMajor, dev));
        CK(cudaDeviceGetAttribute(&st.cc_minor, cudaDevAttrComputeCapabilityMinor, dev));
        st.device = dev;
    }
    if (!(st.cc_major == 10 && st.cc_minor == 3))
        return fail(GNS_ERR_UNSUPPORTED, "this library is built for sm_103a (GB300) only");
    if (!st.err) {
        CK(cudaMalloc(&st.err, 256));
        CK(cudaMemset(st.err, 0, 256));
    }
    const char* cap = std::getenv("GNS_NUM_SMS");
    if (cap && std::atoi(cap) > 0) st.num_sms = std::min(st.num_sms, std::atoi(cap));
    *out = &st;
    return GNS_OK;
}

// Bound of every device-side wait: 2 s, or GNS_WAIT_LIMIT_MS.
unsigned long long wait_limit_ns() {
    const char* e = std::getenv("GNS_WAIT_LIMIT_MS");
    if (e && std::atoll(e) > 0) return static_cast<unsigned long long>(std::atoll(e)) * 1000000ull;
    return kDefaultWaitLimitNs;
}

// Starts a call on a device: a new epoch for its kernels' abort mark.
void begin_call(DeviceState& st) {
    st.epoch = st.epoch == 0x7fffffff ? 1 : st.epoch + 1;
    st.status = DevStatus{st.err, st.epoch, 0, wait_limit_ns()};
}

int ensure_workspace(DeviceState& st, size_t bytes) {
    if (st.ws_bytes >= bytes) return GNS_OK;
    if (st.ws) {
        CK(cudaDeviceSynchronize());
        CK(cudaFree(st.ws));
        st.ws = nullptr;
        st.ws_bytes = 0;
    }
    const size_t want = align_up(bytes, size_t(2) << 20);
    if (cudaMalloc(&st.ws, want) != cudaSuccess) {
        cudaGetLastError();
        st.ws = nullptr;
        return fail(GNS_ERR_NOMEM, "workspace allocation of " + std::to_string(want) + " bytes failed");
    }
    st.ws_bytes = want;
    return GNS_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant of gns_orthogonalize_batched.
//
// Some callers cannot let the library call cudaMalloc: their device memory is
// already held by their own allocator or pool, or they cannot accept the
// device-wide synchronization that growing the cached workspace costs
// (cudaDeviceSynchronize, cudaFree, cudaMalloc). For them the workspace of
// this entry point is one fixed array in device memory, declared below, that
// every GPU which loads the library holds until the process exits.

constexpr size_t kNoAllocBytes = size_t(64) << 20;  // size of the fixed array
constexpr size_t kNoAllocStatusBytes = 256;         // status word, then the workspace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

struct NoAllocDevice {
    bool ready = false;
    char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int num_sms = 0;
    int cc_major = 0, cc_minor = 0;
    int epoch = 0;            // number of the current allocation-free call on this device
};

std::mutex g_noalloc_mu;
std::map<int, NoAllocDevice> g_noalloc;


// ------------------------------------------------------- launch accounting
//
// Every kernel launch is counted. When profiling is on, each launch is also
// bracketed by a pair of CUDA events on its own stream; gns_profile_read()
// turns them into per-class launch counts and summed durations.

enum KernelClass { kClsGemm = 0, kClsNorm = 1, kClsMuon = 2, kClsCopy = 3, kNumCls = 4 };

std::atomic<long long> g_launches{0};
std::atomic<bool> g_profiling{false};
std::mutex g_prof_mu;
struct ProfRec {
    cudaEvent_t a, b;
    int cls;
};
std::vector<ProfRec> g_recs;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return e;
}

template <typename F>
int counted_launch(int cls, cudaStream_t s, F&& fn) {
    ProfRec rec{nullptr, nullptr, cls};
    const bool prof = g_profiling.load();
    if (prof) {
        std::lock_guard<std::mutex> lk(g_prof_mu);
        rec.a = take_event();
        rec.b = take_event();
        if (rec.a) cudaEventRecord(rec.a, s);
    }
    const int r = fn();
    g_launches.fetch_add(1);
    if (prof && rec.a && rec.b) {
        cudaEventRecord(rec.b, s);
        std::lock_guard<std::mutex> lk(g_prof_mu);
        g_recs.push_back(rec);
    }
    return r;
}

#define LAUNCH(cls, call) CK(counted_launch((cls), s, [&]() { return static_cast<int>(call); }))

// ------------------------------------------------------------ tensor maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// A set of G row-major matrices in device memory.
struct Mat {
    void* p = nullptr;
    int rows = 0, cols = 0;
    long long ld = 0, stride = 0;
    bool f32 = false;
};

int make_map(CUtensorMap* m, const Mat& x, int G, uint32_t box_c, uint32_t box_r, CUtensorMapSwizzle sw) {
    auto fn = encode_fn();
    if (!fn) return fail(GNS_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
    const size_t es = x.f32 ? 4 : 2;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(x.cols), static_cast<cuuint64_t>(x.rows),
                          static_cast<cuuint64_t>(G)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(x.ld) * es, static_cast<cuuint64_t>(x.stride) * es};
    cuuint32_t box[3] = {box_c, box_r, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, x.f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, x.p, dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char buf[256];
        std::snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled failed (%d): %d x %d, ld %lld, G %d", static_cast<int>(r),
                      x.rows, x.cols, x.ld, G);
        return fail(GNS_ERR_INVALID, buf);
    }
    return GNS_OK;
}

// One problem of a phase: D = alpha A B^T (+ beta C) [, D2 = delta D + gamma I].
// A is M x K, B is N x K. An operand marked MN-major is given by its stored
// transpose (A: K x M, B: K x N, row-major) and read through the transposed
// descriptor, so no transposed copy is ever materialized.
struct ProblemSpec {
    Mat A, B, D;
    bool a_mn = false, b_mn = false;
    const Mat* C = nullptr;
    const Mat* Dt = nullptr;
    const Mat* D2 = nullptr;
    const Mat* D2t = nullptr;
    float alpha = 1.f, beta = 0.f, delta = 0.f, gamma = 0.f;
    bool sym = false;
    // Lower-only storage of symmetric matrices (square tile shapes only):
    // A / B are read that way, D (and D2) are written that way.
    bool a_sym = false, b_sym = false, lower = false;
    const MuonFuse* muon = nullptr;  // fused Muon update instead of storing D
};

// Tile shape for a program: 256 x 256 tiles on CTA pairs when the matrices
// fill them; else 128 x 128 tiles on single CTAs.
// GNS_TILE=128x1|256x1|256x2 forces one shape (tuning).
struct TileShape {
    int bn, cg;
};

TileShape choose_tile(int n, int G, int num_sms) {
    const char* force = std::getenv("GNS_TILE");
    if (force) {
        const std::string f(force);
        if (f == "128x1") return {128, 1};
        if (f == "256x1") return {256, 1};
        if (f == "256x2") return {256, 2};
    }
    if (n < 192) return {128, 1};
    // A bucket whose n x n products give the CTA pairs less than about one and
    // a half waves of 256 x 256 tiles leaves pairs idle: single-CTA 128 x 128
    // tiles quadruple the tile count (measured: 16 x 256 x 4096, 32 x 384 x 1536
    // and 8 x 512 x 2048 run 15-17 % faster that way, 24 x 1024 x 4096 and
    // 256 x 512 x 2048 slower).
    const long long t2 = (n + 255) / 256;
    const long long pair_tiles = static_cast<long long>(G) * t2 * (t2 + 1) / 2;
    if (2 * pair_tiles < 3LL * (num_sms / 2)) return {128, 1};
    return {256, 2};
}

bool self_sym() {
    const char* e = std::getenv("GNS_SELF_SYM");
    return !(e && std::atoi(e) == 0);
}

// Full-width output blocks are stored straight from registers unless
// GNS_DIRECT_STORE=0 (staged through shared memory).
bool direct_store() {
    const char* e = std::getenv("GNS_DIRECT_STORE");
    return !(e && std::atoi(e) == 0);
}

// How many tiles ahead of its producer a CTA pair claims (GNS_LOOKAHEAD,
// 1 .. 8; default 1): enough to hide the claim, the decode and the
// dependency acquire, few enough that no CTA holds tiles another CTA could
// start sooner.
int lookahead() {
    const char* e = std::getenv("GNS_LOOKAHEAD");
    const int v = e ? std::atoi(e) : 1;
    return v < 1 ? 1 : (v > 8 ? 8 : v);
}

// Non-symmetric products walk their tiles column by column unless
// GNS_COL_WALK=0 (row by row).
bool col_walk() {
    const char* e = std::getenv("GNS_COL_WALK");
    return !(e && std::atoi(e) == 0);
}

// Collects the phases of one launch. Tensor maps are shared between the
// problems that read or write the same buffer with the same box.
//
// The launch's work list (see gemm.cuh) is numbered here: each phase gets
// its first ticket and the counter target of its tiles (the signals of
// every earlier tile of the same matrix).
class ProgramBuilder {
  public:
    // sync: 1 + G ints in device memory, the launch's ticket counter
    // followed by the per-matrix counters.
    ProgramBuilder(DeviceState& st, int G, TileShape ts, int* sync, cudaStream_t s)
        : st_(st), G_(G), ts_(ts), sync_(sync), s_(s) {
        reset();
    }

    // Adds a phase of one or two independent problems; launches first when
    // the program is full (the next launch then depends on it by stream order).
    int phase(const ProblemSpec& p0, const ProblemSpec* p1) {
        const int need_probs = p1 ? 2 : 1;
        if (prog_.nphase + 1 > kMaxPhases || prog_.nprob + need_probs > kMaxProblems || prog_.nmaps + 8 > kMaxMaps)
            RET(flush());
        GemmPhaseDesc& ph = prog_.phase[prog_.nphase];
        ph.prob_begin = prog_.nprob;
        ph.nprob = 0;
        ph.tiles_per_matrix = 0;
        for (const ProblemSpec* sp : {&p0, p1}) {
            if (!sp) continue;
            GemmProblem& pr = prog_.prob[prog_.nprob];
            RET(set_problem(pr, *sp));
            ph.tiles_per_matrix += pr.tiles_per_matrix;
            ph.nprob += 1;
            prog_.nprob += 1;
        }
        const long long spi = gemm_signals_per_tile(ts_.cg);
        const long long per = ph.tiles_per_matrix;
        if (items_done_ + per * G_ > (1LL << 30) || signals_done_ + per * spi > (1LL << 30))
            return fail(GNS_ERR_INVALID, "program too large for one launch");
        ph.item_begin = static_cast<int>(items_done_);
        ph.wait = static_cast<int>(signals_done_);
        items_done_ += per * G_;
        signals_done_ += per * spi;
        prog_.total_items = static_cast<int>(items_done_);
        prog_.nphase += 1;
        return GNS_OK;
    }

    // The caller cleared the counters for the next launch (stream-ordered).
    void counters_cleared() { cleared_ = true; }

    int flush() {
        if (prog_.nphase == 0) return GNS_OK;
        // The ticket counter and the matrices' counters start at zero.
        if (!cleared_) CK(cudaMemsetAsync(sync_, 0, sizeof(int) * (1 + static_cast<size_t>(G_)), s_));
        prog_.ticket = sync_;
        prog_.counters = prog_.nphase > 1 ? sync_ + 1 : nullptr;
        prog_.direct_store = direct_store() ? 1 : 0;
        prog_.lookahead = lookahead();
        prog_.st = st_.status;
        prog_.G = G_;
        cudaStream_t s = s_;
        LAUNCH(kClsGemm, launch_gemm_program(prog_, ts_.bn, ts_.cg, st_.num_sms, s));
        reset();
        cleared_ = false;
        return GNS_OK;
    }

  private:
    void reset() {
        std::memset(&prog_, 0, sizeof(prog_));
        keys_.clear();
        items_done_ = 0;
        signals_done_ = 0;
    }

    int map_index(const Mat& x, uint32_t box_c, uint32_t box_r, CUtensorMapSwizzle sw) {
        const std::string key = std::to_string(reinterpret_cast<uintptr_t>(x.p)) + ":" + std::to_string(x.rows) + ":" +
                                std::to_string(x.cols) + ":" + std::to_string(x.ld) + ":" + std::to_string(x.stride) +
                                ":" + std::to_string(x.f32) + ":" + std::to_string(box_c) + ":" +
                                std::to_string(box_r) + ":" + std::to_string(static_cast<int>(sw));
        for (size_t i = 0; i < keys_.size(); ++i)
            if (keys_[i] == key) return static_cast<int>(i);
        if (prog_.nmaps >= kMaxMaps) return -1;
        if (make_map(&prog_.maps[prog_.nmaps], x, G_, box_c, box_r, sw) != GNS_OK) return -2;
        keys_.push_back(key);
        return prog_.nmaps++;
    }

    // K-major: box {64 (K), rows per CTA} (A: 128, B: bn / cg). MN-major: box
    // {64 (M or N), 64 (K)} over the stored transpose.
    int operand(const Mat& x, uint32_t box_rows, int& idx, bool mn) {
        (void)mn;
        idx = map_index(x, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
        return idx >= 0 ? GNS_OK : (idx == -1 ? fail(GNS_ERR_INVALID, "tensor map table full") : GNS_ERR_INVALID);
    }

    // Outputs are written by the epilogue's own stores in 16-byte pieces.
    static int output(const Mat& x, OutView& o) {
        const size_t es = x.f32 ? 4 : 2;
        if (reinterpret_cast<uintptr_t>(x.p) % 16 != 0 || (x.ld * es) % 16 != 0 || (x.stride * es) % 16 != 0)
            return fail(GNS_ERR_INVALID, "outputs need 16-byte aligned rows");
        o.p = x.p;
        o.ld = x.ld;
        o.stride = x.stride;
        return GNS_OK;
    }

    int set_problem(GemmProblem& pr, const ProblemSpec& sp) {
        std::memset(&pr, 0, sizeof(pr));
        const int bn = ts_.bn, cg = ts_.cg;
        const int M = sp.a_mn ? sp.A.cols : sp.A.rows, Ka = sp.a_mn ? sp.A.rows : sp.A.cols;
        const int N = sp.b_mn ? sp.B.cols : sp.B.rows, Kb = sp.b_mn ? sp.B.rows : sp.B.cols;
        if (Ka != Kb) return fail(GNS_ERR_INVALID, "operand K mismatch");
        if (sp.sym && M != N) return fail(GNS_ERR_INVALID, "symmetric product must be square");
        if (sp.D2 && sp.Dt && !sp.D2t) return fail(GNS_ERR_INVALID, "second output needs its transposed map");
        if (sp.D.f32 && (sp.Dt || sp.D2)) return fail(GNS_ERR_INVALID, "fp32 output supports no transposed/second output");
        if (G_ > 65535) return fail(GNS_ERR_INVALID, "too many matrices in one launch");
        pr.mA = pr.mB = pr.mC = pr.mAt = pr.mBt = -1;
        if ((sp.a_sym || sp.b_sym || sp.lower) && bn != 128 * cg)
            return fail(GNS_ERR_INVALID, "lower-only storage needs square tiles");
        if ((sp.a_sym && sp.a_mn) || (sp.b_sym && sp.b_mn)) return fail(GNS_ERR_INVALID, "lower-only operands are K-major");
        RET(operand(sp.A, sp.a_mn ? 64u : 128u, pr.mA, sp.a_mn));
        RET(operand(sp.B, sp.b_mn ? 64u : static_cast<uint32_t>(bn / cg), pr.mB, sp.b_mn));
        if (sp.muon) {
            if (sp.sym || sp.Dt || sp.D2) return fail(GNS_ERR_INVALID, "the fused update needs a plain product");
            pr.muon = *sp.muon;
        } else {
            RET(output(sp.D, pr.d));
        }
        int flags = 0;
        if (sp.sym) flags |= kFlagSym;
        if (sp.D.f32) flags |= kFlagOutF32;
        if (sp.a_mn) flags |= kFlagAmn;
        if (sp.b_mn) flags |= kFlagBmn;
        if (sp.a_sym) {
            flags |= kFlagAsym;
            RET(operand(sp.A, 64u, pr.mAt, true));
        }
        if (sp.b_sym) {
            flags |= kFlagBsym;
            RET(operand(sp.B, 64u, pr.mBt, true));
        }
        if (sp.lower) flags |= kFlagLower;
        if (sp.muon) flags |= kFlagMuon;
        if (!sp.sym && col_walk()) flags |= kFlagColWalk;
        // A symmetric product of one stored matrix with itself (X X^T, R R,
        // A A): with an exactly symmetric addend, its diagonal tiles are
        // exactly symmetric as computed (GNS_SELF_SYM=0 mirrors them instead).
        if (sp.sym && sp.A.p == sp.B.p && sp.A.ld == sp.B.ld && sp.A.stride == sp.B.stride && sp.A.rows == sp.B.rows &&
            sp.A.cols == sp.B.cols && sp.a_mn == sp.b_mn && sp.a_sym == sp.b_sym && self_sym())
            flags |= kFlagSelfSym;
        if (sp.C) {
            flags |= kFlagC;
            pr.C = static_cast<const __half*>(sp.C->p);
            pr.ldc = sp.C->ld;
            pr.strideC = sp.C->stride;
            // The epilogue reads C in 32 x 32 blocks by TMA.
            pr.mC = map_index(*sp.C, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
            if (pr.mC < 0) return pr.mC == -1 ? fail(GNS_ERR_INVALID, "tensor map table full") : GNS_ERR_INVALID;
        }
        if (sp.Dt) {
            flags |= kFlagDt;
            RET(output(*sp.Dt, pr.dt));
        }
        if (sp.D2) {
            flags |= kFlagD2;
            RET(output(*sp.D2, pr.d2));
            if (sp.D2t) RET(output(*sp.D2t, pr.d2t));
        }
        pr.alpha = sp.alpha;
        pr.beta = sp.beta;
        pr.delta = sp.delta;
        pr.gamma = sp.gamma;
        pr.M = M;
        pr.N = N;
        pr.K = Ka;
        pr.tiles_n = (pr.N + bn - 1) / bn;
        pr.tiles_m = (pr.M + 128 * cg - 1) / (128 * cg);
        pr.tiles_per_matrix = gemm_tiles_per_matrix(pr.M, pr.N, bn, cg, sp.sym, &pr.tiles_n_walk);
        pr.flags = flags;
        return GNS_OK;
    }

    DeviceState& st_;
    int G_;
    TileShape ts_;
    int* sync_;
    cudaStream_t s_;
    GemmProgram prog_;
    bool cleared_ = false;
    std::vector<std::string> keys_;
    long long items_done_ = 0;    // list items of the phases added so far
    long long signals_done_ = 0;  // counter signals per matrix of those phases
};

// --------------------------------------------------------------- planner

int ilog2(int v) {
    int r = 0;
    while ((1 << (r + 1)) <= v) ++r;
    return r;
}

struct Coeffs {
    std::vector<float> a, b, c;
};

int load_coeffs(const float* coeffs, int steps, Coeffs& out) {
    out.a.resize(steps);
    out.b.resize(steps);
    out.c.resize(steps);
    for (int t = 0; t < steps; ++t) {
        const float* src = coeffs ? coeffs + 3 * t : kQuintic;
        if (!std::isfinite(src[0]) || !std::isfinite(src[1]) || !std::isfinite(src[2]))
            return fail(GNS_ERR_INVALID, "non-finite coefficient");
        out.a[t] = src[0];
        out.b[t] = src[1];
        out.c[t] = src[2];
    }
    return GNS_OK;
}

// Restart schedules as bit masks: bit t set = restart after step t
// (1 <= t < steps). The periodic schedule restarts after every multiple of
// restart_at that leaves at least one full period (Dion3 Algorithm 3: T = 5,
// restart_at = 2 restarts once, after step 2).
uint64_t periodic_restarts(int steps, int restart_at) {
    uint64_t m = 0;
    if (restart_at <= 0) return 0;
    for (int t = 1; t < steps; ++t)
        if (t % restart_at == 0 && steps - t >= restart_at) m |= uint64_t(1) << t;
    return m;
}

bool is_restart_after(int t, int steps, uint64_t restarts) {
    return t >= 1 && t < steps && ((restarts >> t) & 1);
}

// Where the result of one bucket goes.
struct OutSpec {
    Mat out;        // fp32 [G][R][C] (ABI) or fp16 [G][R][ld] (Muon O)
    const MuonFuse* muon = nullptr;  // set: the last product updates W instead of storing out
    bool copy_back = false;  // out is a workspace buffer; copy to user_ptr afterwards
    float* user_ptr = nullptr;
};

struct BucketGeom {
    int R, C, n, m;
    bool transposed, square;
    long long ldn, ldm;
    int k_exp;
    float s;  // 4^k
};

BucketGeom make_geom(int R, int C) {
    BucketGeom g;
    g.R = R;
    g.C = C;
    g.n = std::min(R, C);
    g.m = std::max(R, C);
    g.transposed = R > C;
    g.square = R == C;
    g.ldn = round_up_ll(g.n, 8);
    g.ldm = round_up_ll(g.m, 8);
    g.k_exp = std::min(6, ilog2(g.n) / 2);
    g.s = std::ldexp(1.0f, 2 * g.k_exp);
    return g;
}

// Workspace layout for a chunk of Gc matrices. The fp16 copies of X keep the
// input's own orientation (R x C): Xa holds X0 (and the standard-NS iterates
// alternate between Xa and Xb), Xb holds X after the restart.
struct Layout {
    size_t xa, xb, r, z, rz, qa, qb, partial, queue, sync, sync_bytes, out32, o16, meta, total;
    long long ld_x;
    long long ld_out32;
};

Layout make_layout(const BucketGeom& g, int Gc, bool need_out32, bool need_o16, size_t meta_bytes) {
    Layout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    L.ld_x = round_up_ll(g.C, 8);
    const size_t xs = static_cast<size_t>(g.R) * L.ld_x * 2 * Gc;
    const size_t nn = static_cast<size_t>(g.n) * g.ldn * 2 * Gc;
    L.xa = take(xs);
    L.xb = take(xs);
    L.r = take(nn);
    L.z = take(nn);
    L.rz = g.square ? 0 : take(nn);
    L.qa = g.square ? 0 : take(nn);
    L.qb = g.square ? 0 : take(nn);
    L.partial = take(static_cast<size_t>(Gc) * norm_parts(static_cast<long long>(g.R) * g.C) * 4);
    // The norm/cast queue (1 + Gc ints), then the GEMM program's ticket and
    // per-matrix counters (1 + Gc ints): adjacent, so that one clear covers
    // both.
    L.sync_bytes = (2 + 2 * static_cast<size_t>(Gc)) * 4;
    L.queue = take(L.sync_bytes);
    L.sync = L.queue + (1 + static_cast<size_t>(Gc)) * 4;
    L.ld_out32 = round_up_ll(g.C, 4);
    L.out32 = need_out32 ? take(static_cast<size_t>(g.R) * L.ld_out32 * 4 * Gc) : 0;
    L.o16 = need_o16 ? take(static_cast<size_t>(g.R) * round_up_ll(g.C, 8) * 2 * Gc) : 0;
    L.meta = take(meta_bytes);
    L.total = off;
    return L;
}

Mat mat16(char* ws, size_t off, int rows, int cols, long long ld) {
    Mat m;
    m.p = ws + off;
    m.rows = rows;
    m.cols = cols;
    m.ld = ld;
    m.stride = static_cast<long long>(rows) * ld;
    m.f32 = false;
    return m;
}

// Where a run left its Gram state (rectangular buckets): the last R it
// computed and the final Q, each Gc fp16 n x n matrices (row stride ld,
// matrix stride stride, elements); stored R = s R (s = 4^k), Q unscaled.
struct GramState {
    const void* r = nullptr;
    const void* q = nullptr;
    long long ld = 0, stride = 0;
    float s = 1.0f;
};

// Runs the orthogonalization of one chunk of Gc fp32 matrices `in` (the
// momentum, first updated in place as M <- mu M + G, when grads is given).
int run_core(DeviceState& st, const BucketGeom& g, const Layout& L, int Gc, const MatrixSet& in,
             const MatrixSet* grads, float mu, int steps, uint64_t restarts, const Coeffs& cf, const OutSpec& os,
             cudaStream_t s, GramState* state = nullptr) {
    const TileShape ts = choose_tile(g.n, Gc, st.num_sms);
    char* ws = st.ws;
    ProgramBuilder prog(st, Gc, ts, reinterpret_cast<int*>(ws + L.sync), s);
    // Symmetric n x n intermediates are stored lower-only (diagonal tiles in
    // full) when the tiles are square.
    const bool lo = ts.bn == 128 * ts.cg;
    const int n = g.n;
    // Stored copies of X in the input's orientation (R x C).
    Mat Xa = mat16(ws, L.xa, g.R, g.C, L.ld_x);
    Mat Xb = mat16(ws, L.xb, g.R, g.C, L.ld_x);
    // The norm/cast queue and the GEMM counters start at zero (the whole
    // region: a last, smaller chunk still uses the layout's offsets).
    CK(cudaMemsetAsync(ws + L.queue, 0, L.sync_bytes, s));
    prog.counters_cleared();
    {
        // Norm, scale and fp16 cast (with the momentum update first, for the
        // Muon step), right before the GEMM program.
        NormCastJob job{};
        job.in = in;
        if (grads) job.grads = *grads;
        job.mu = mu;
        job.G = Gc;
        job.R = g.R;
        job.C = g.C;
        job.k_exp = g.k_exp;
        job.out = Xa.p;
        job.ld_out = Xa.ld;
        job.stride_out = Xa.stride;
        job.partial = reinterpret_cast<float*>(ws + L.partial);
        job.queue = reinterpret_cast<int*>(ws + L.queue);
        job.st = st.status;
        LAUNCH(kClsNorm, launch_norm_cast(job, st.num_sms, s));
    }
    const float inv_s = 1.0f / g.s;
    const float out_scale = std::ldexp(1.0f, -g.k_exp);
    // Operand views of the stored X (Xs = X when R <= C, Xs = X^T when R > C):
    // X as an n-row operand (K = m) and X^T as an m-row operand (K = n).
    auto x_rows = [&](ProblemSpec& p, bool as_a, const Mat& xs) {
        (as_a ? p.A : p.B) = xs;
        (as_a ? p.a_mn : p.b_mn) = g.transposed;
    };
    auto xt_rows = [&](ProblemSpec& p, bool as_a, const Mat& xs) {
        (as_a ? p.A : p.B) = xs;
        (as_a ? p.a_mn : p.b_mn) = !g.transposed;
    };
    auto phase = [&](const ProblemSpec& p0, const ProblemSpec* p1) { return prog.phase(p0, p1); };

    if (g.square) {
        // Dion3 Algorithm 1 with symmetric A = X X^T and B = b A + c A^2
        // (App. C.3): X <- a X + B X, the last step writing the output.
        Mat A = mat16(ws, L.r, n, n, g.ldn);
        Mat B = mat16(ws, L.z, n, n, g.ldn);
        Mat X = Xa, Xn = Xb;
        for (int t = 0; t < steps; ++t) {
            ProblemSpec pa;
            x_rows(pa, true, X);
            x_rows(pa, false, X);
            pa.D = A;
            pa.Dt = &A;
            pa.sym = true;
            pa.lower = lo;
            RET(phase(pa, nullptr));
            ProblemSpec pb;
            pb.A = A;
            pb.B = A;
            pb.C = &A;
            pb.D = B;
            pb.Dt = &B;
            pb.alpha = cf.c[t] * inv_s;
            pb.beta = cf.b[t];
            pb.sym = true;
            pb.a_sym = pb.b_sym = pb.lower = lo;
            RET(phase(pb, nullptr));
            // X' = B X + a X: B is symmetric, X enters as the N x K operand X^T.
            ProblemSpec px;
            px.A = B;
            px.a_sym = lo;
            xt_rows(px, false, X);
            px.C = &X;
            if (t + 1 < steps) {
                px.D = Xn;
                px.alpha = inv_s;
                px.beta = cf.a[t];
                RET(phase(px, nullptr));
                std::swap(X, Xn);
            } else {
                px.D = os.out;
                px.muon = os.muon;
                px.alpha = inv_s * out_scale;
                px.beta = cf.a[t] * out_scale;
                RET(phase(px, nullptr));
            }
        }
        return prog.flush();
    }

    // Dion3 Algorithm 3 with the App. B.2.3 a-term distribution.
    Mat R = mat16(ws, L.r, n, n, g.ldn);
    Mat Z = mat16(ws, L.z, n, n, g.ldn);
    Mat RZ = mat16(ws, L.rz, n, n, g.ldn);
    Mat Qc = mat16(ws, L.qa, n, n, g.ldn);
    Mat Qn = mat16(ws, L.qb, n, n, g.ldn);
    Mat X = Xa, Xn = Xb;

    auto gram = [&](void) -> int {
        ProblemSpec p;
        x_rows(p, true, X);
        x_rows(p, false, X);
        p.D = R;
        p.Dt = &R;
        p.sym = true;
        p.lower = lo;
        return phase(p, nullptr);
    };
    // Q X in the stored orientation: Q X (R <= C) or X^T Q = (Q X)^T (R > C).
    auto qx = [&](ProblemSpec& p) {
        if (!g.transposed) {
            p.A = Qc;
            p.a_sym = lo;
            xt_rows(p, false, X);
        } else {
            xt_rows(p, true, X);
            p.B = Qc;
            p.b_sym = lo;
        }
    };
    RET(gram());
    bool q_identity = true;
    for (int t = 1; t <= steps; ++t) {
        const float a = cf.a[t - 1], b = cf.b[t - 1], c = cf.c[t - 1];
        if (is_restart_after(t - 1, steps, restarts)) {
            // X <- Q X, then R <- X X^T, Q <- I.
            ProblemSpec p;
            qx(p);
            p.D = Xn;
            RET(phase(p, nullptr));
            std::swap(X, Xn);
            RET(gram());
            q_identity = true;
        }
        const bool need_r = t < steps && !is_restart_after(t, steps, restarts);
        // Z = b R + c R^2 (with Q = Z + a I written alongside after a (re)start).
        {
            ProblemSpec p;
            p.A = R;
            p.B = R;
            p.C = &R;
            p.D = Z;
            p.Dt = &Z;
            p.alpha = c * inv_s;
            p.beta = b;
            p.sym = true;
            p.a_sym = p.b_sym = p.lower = lo;
            if (q_identity) {
                p.D2 = &Qc;
                p.D2t = &Qc;
                p.delta = inv_s;
                p.gamma = a;
            }
            RET(phase(p, nullptr));
        }
        ProblemSpec pq, prz;
        if (!q_identity) {
            pq.A = Qc;
            pq.B = Z;
            pq.C = &Qc;
            pq.D = Qn;
            pq.Dt = &Qn;
            pq.alpha = inv_s;
            pq.beta = a;
            pq.sym = true;
            pq.a_sym = pq.b_sym = pq.lower = lo;
        }
        if (need_r) {
            prz.A = R;
            prz.B = Z;
            prz.C = &R;
            prz.D = RZ;
            prz.Dt = &RZ;
            prz.alpha = inv_s;
            prz.beta = a;
            prz.sym = true;
            prz.a_sym = prz.b_sym = prz.lower = lo;
        }
        if (!q_identity && need_r) {
            RET(phase(pq, &prz));
        } else if (!q_identity) {
            RET(phase(pq, nullptr));
        } else if (need_r) {
            RET(phase(prz, nullptr));
        }
        if (!q_identity) std::swap(Qc, Qn);
        q_identity = false;
        if (need_r) {
            ProblemSpec p;
            p.A = Z;
            p.B = RZ;
            p.C = &RZ;
            p.D = R;
            p.Dt = &R;
            p.alpha = inv_s;
            p.beta = a;
            p.sym = true;
            p.a_sym = p.b_sym = p.lower = lo;
            RET(phase(p, nullptr));
        }
    }
    if (state) {
        state->r = R.p;
        state->q = Qc.p;
        state->ld = R.ld;
        state->stride = R.stride;
        state->s = g.s;
    }
    // O = Q X, written in the caller's orientation.
    ProblemSpec p;
    qx(p);
    p.D = os.out;
    p.muon = os.muon;
    p.alpha = out_scale;
    RET(phase(p, nullptr));
    return prog.flush();
}

size_t chunk_cap_bytes() {
    const char* e = std::getenv("GNS_WORKSPACE_CAP_MB");
    if (e && std::atoll(e) > 0) return static_cast<size_t>(std::atoll(e)) << 20;
    return size_t(24) << 30;
}

int validate_common(int G, int R, int C, int steps) {
    if (G < 0 || R < 1 || C < 1) return fail(GNS_ERR_INVALID, "G must be >= 0 and R, C >= 1");
    if (steps < 1 || steps > GNS_MAX_STEPS) return fail(GNS_ERR_INVALID, "steps must be in 1..GNS_MAX_STEPS");
    if (static_cast<long long>(R) * C > (1LL << 40)) return fail(GNS_ERR_INVALID, "matrix too large");
    return GNS_OK;
}

int chunk_size(const BucketGeom& g, int G, bool out32, bool o16) {
    const Layout one = make_layout(g, 1, out32, o16, 0);
    size_t per = one.total;
    size_t cap = chunk_cap_bytes();
    long long c = static_cast<long long>(cap / std::max<size_t>(per, 1));
    if (c < 1) c = 1;
    if (c > G) c = G;
    if (c > 65535) c = 65535;
    return static_cast<int>(c);
}

int orthogonalize_device(float* ptr, int G, int R, int C, int steps, uint64_t restarts, const float* coeffs,
                         cudaStream_t s) {
    RET(validate_common(G, R, C, steps));
    if (G == 0) return GNS_OK;
    if (!ptr) return fail(GNS_ERR_INVALID, "ptr is null");
    DeviceState* st = nullptr;
    RET(get_state(&st));
    begin_call(*st);
    Coeffs cf;
    RET(load_coeffs(coeffs, steps, cf));
    const BucketGeom g = make_geom(R, C);
    const bool direct_out = (reinterpret_cast<uintptr_t>(ptr) % 16 == 0) && ((static_cast<long long>(C) * 4) % 16 == 0);
    const int Gc = chunk_size(g, G, !direct_out, false);
    const Layout L = make_layout(g, Gc, !direct_out, false, 0);
    RET(ensure_workspace(*st, L.total));
    const long long numel = static_cast<long long>(R) * C;
    for (int g0 = 0; g0 < G; g0 += Gc) {
        const int gc = std::min(Gc, G - g0);
        float* base = ptr + static_cast<long long>(g0) * numel;
        MatrixSet in{base, numel, nullptr};
        OutSpec os;
        if (direct_out) {
            os.out.p = base;
            os.out.rows = R;
            os.out.cols = C;
            os.out.ld = C;
            os.out.stride = numel;
            os.out.f32 = true;
        } else {
            os.out.p = st->ws + L.out32;
            os.out.rows = R;
            os.out.cols = C;
            os.out.ld = L.ld_out32;
            os.out.stride = static_cast<long long>(R) * L.ld_out32;
            os.out.f32 = true;
        }
        RET(run_core(*st, g, L, gc, in, nullptr, 0.0f, steps, restarts, cf, os, s));
        if (!direct_out)
            LAUNCH(kClsCopy, launch_copy_rows_f32(static_cast<float*>(os.out.p), os.out.ld, os.out.stride, base, gc, R, C, s));
    }
    return GNS_OK;
}

// The Muon update runs in the epilogue of the last product (the default), or
// as a separate pass over a stored fp16 O when GNS_MUON_FUSED=0; both give
// identical bits.
bool muon_fused() {
    const char* e = std::getenv("GNS_MUON_FUSED");
    return !(e && std::string(e) == "0");
}

// One Muon (vm == nullptr) or NorMuon step over n matrices, bucketed by shape.
int optimizer_step(const gns_tensor* params, const gns_tensor* grads, const gns_tensor* momentum,
                   const gns_tensor* vm, int n, float lr, float wd, float mu, float beta2, float eps, uint64_t seed,
                   uint64_t step, void* stream) {
    if (n < 0) return fail(GNS_ERR_INVALID, "n < 0");
    if (n == 0) return GNS_OK;
    if (!params || !grads || !momentum) return fail(GNS_ERR_INVALID, "null tensor array");
    for (int i = 0; i < n; ++i) {
        const gns_tensor &w = params[i], &gr = grads[i], &mm = momentum[i];
        if (!w.data || !gr.data || !mm.data) return fail(GNS_ERR_INVALID, "null tensor data");
        if (w.rows < 1 || w.cols < 1 || gr.rows != w.rows || gr.cols != w.cols || mm.rows != w.rows ||
            mm.cols != w.cols)
            return fail(GNS_ERR_INVALID, "tensor shapes differ");
        if (w.base_index < 0) return fail(GNS_ERR_INVALID, "negative base_index");
        if (vm && (!vm[i].data || vm[i].rows != w.rows || vm[i].cols != 1))
            return fail(GNS_ERR_INVALID, "second moments must be rows x 1");
    }
    if (vm && !(beta2 >= 0.0f && beta2 <= 1.0f && eps >= 0.0f)) return fail(GNS_ERR_INVALID, "bad beta2 or eps");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DeviceState* st = nullptr;
    RET(get_state(&st));
    begin_call(*st);
    // Buckets of equal (rows, cols), in order of first appearance.
    std::vector<std::pair<std::pair<int, int>, std::vector<int>>> buckets;
    for (int i = 0; i < n; ++i) {
        auto key = std::make_pair(params[i].rows, params[i].cols);
        auto it = std::find_if(buckets.begin(), buckets.end(), [&](const auto& b) { return b.first == key; });
        if (it == buckets.end()) {
            buckets.push_back({key, {i}});
        } else {
            it->second.push_back(i);
        }
    }
    Coeffs cf;
    RET(load_coeffs(nullptr, 5, cf));
    const int narr = vm ? 4 : 3;  // pointer arrays: M, G, W (, V)
    for (auto& bk : buckets) {
        const int R = bk.first.first, C = bk.first.second;
        const int G = static_cast<int>(bk.second.size());
        const BucketGeom g = make_geom(R, C);
        // NorMuon needs all of O before its row statistics: it stores O.
        const bool fused = !vm && muon_fused();
        const size_t per_matrix_meta = narr * sizeof(void*) + sizeof(long long) + (vm ? 4 * sizeof(float) * R : 0);
        int Gc = chunk_size(g, G, false, !fused);
        // The statistics buffers live in the metadata block.
        while (Gc > 1 && make_layout(g, Gc, false, !fused, static_cast<size_t>(Gc) * per_matrix_meta + 1024).total >
                             chunk_cap_bytes())
            --Gc;
        const size_t meta_bytes = static_cast<size_t>(Gc) * per_matrix_meta + 1024;
        const Layout L = make_layout(g, Gc, false, !fused, meta_bytes);
        RET(ensure_workspace(*st, L.total));
        const long long ld_o = round_up_ll(C, 8);
        const float scale = 0.2f * std::sqrt(static_cast<float>(std::max(R, C)));
        for (int g0 = 0; g0 < G; g0 += Gc) {
            const int gc = std::min(Gc, G - g0);
            std::vector<const void*> ptrs(narr * static_cast<size_t>(gc));
            std::vector<long long> bases(gc);
            for (int j = 0; j < gc; ++j) {
                const int i = bk.second[g0 + j];
                ptrs[j] = momentum[i].data;
                ptrs[gc + j] = grads[i].data;
                ptrs[2 * gc + j] = params[i].data;
                if (vm) ptrs[3 * gc + j] = vm[i].data;
                bases[j] = params[i].base_index;
            }
            char* meta = st->ws + L.meta;
            CK(cudaMemcpyAsync(meta, ptrs.data(), ptrs.size() * sizeof(void*), cudaMemcpyHostToDevice, s));
            long long* bases_dev = reinterpret_cast<long long*>(meta + align_up(ptrs.size() * sizeof(void*), 16));
            CK(cudaMemcpyAsync(bases_dev, bases.data(), bases.size() * sizeof(long long), cudaMemcpyHostToDevice, s));
            float* stats = reinterpret_cast<float*>(
                meta + align_up(align_up(ptrs.size() * sizeof(void*), 16) + bases.size() * sizeof(long long), 256));
            const void* const* pm = reinterpret_cast<const void* const*>(meta);
            MatrixSet Ms{nullptr, 0, pm};
            MatrixSet Gs{nullptr, 0, pm + gc};
            MatrixSet Ws{nullptr, 0, pm + 2 * gc};
            OutSpec os;
            os.out.rows = R;
            os.out.cols = C;
            os.out.f32 = false;
            MuonFuse mf{};
            if (fused) {
                mf.w = reinterpret_cast<uint16_t* const*>(meta) + 2 * gc;
                mf.base = bases_dev;
                mf.lr = lr;
                mf.wd = wd;
                mf.scale = scale;
                mf.seed_lo = static_cast<uint32_t>(seed);
                mf.seed_hi = static_cast<uint32_t>(seed >> 32);
                mf.step_lo = static_cast<uint32_t>(step);
                mf.step_hi = static_cast<uint32_t>(step >> 32);
                os.muon = &mf;
            } else {
                os.out.p = st->ws + L.o16;
                os.out.ld = ld_o;
                os.out.stride = static_cast<long long>(R) * ld_o;
            }
            RET(run_core(*st, g, L, gc, Ms, &Gs, mu, 5, periodic_restarts(5, 2), cf, os, s));
            if (fused) continue;
            MatrixSet Os{os.out.p, os.out.stride, nullptr};
            const float* row_step = nullptr;
            if (vm) {
                // Dion3 Eq. 2: row second moments, then one factor per matrix.
                MatrixSet Vs{nullptr, 0, pm + 3 * gc};
                const size_t rc = static_cast<size_t>(gc) * R;
                float* row_sq = stats;
                float* row_hat = stats + rc;
                float* inv = stats + 2 * rc;
                float* steps = stats + 3 * rc;
                LAUNCH(kClsMuon, launch_normuon_rows(Os, ld_o, Vs, gc, R, C, beta2, eps, row_sq, row_hat, inv, s));
                LAUNCH(kClsMuon, launch_normuon_factor(row_sq, row_hat, inv, gc, R, lr * scale, steps, s));
                row_step = steps;
            }
            LAUNCH(kClsMuon, launch_muon_update(Ws, Os, ld_o, bases_dev, 0, gc, R, C, lr, wd, scale, seed, step,
                                                st->num_sms, s,
                                                row_step));
        }
    }
    return GNS_OK;
}


// One Dion3 step (Algorithm 4, Muon flavor) over n matrices, bucketed by
// shape: accumulate and rank, gather the selected rows (or columns), run the
// Gram NS core on the k x m submatrices, then update W and damp M.
int dion3_step_impl(const gns_tensor* params, const gns_tensor* grads, const gns_tensor* momentum, int n,
                    float fraction, float lr, float wd, float mu, uint64_t seed, uint64_t step, void* stream) {
    if (n < 0) return fail(GNS_ERR_INVALID, "n < 0");
    if (n == 0) return GNS_OK;
    if (!params || !grads || !momentum) return fail(GNS_ERR_INVALID, "null tensor array");
    if (!(fraction > 0.0f && fraction <= 1.0f)) return fail(GNS_ERR_INVALID, "fraction must be in (0, 1]");
    for (int i = 0; i < n; ++i) {
        const gns_tensor &w = params[i], &gr = grads[i], &mm = momentum[i];
        if (!w.data || !gr.data || !mm.data) return fail(GNS_ERR_INVALID, "null tensor data");
        if (w.rows < 1 || w.cols < 1 || gr.rows != w.rows || gr.cols != w.cols || mm.rows != w.rows ||
            mm.cols != w.cols)
            return fail(GNS_ERR_INVALID, "tensor shapes differ");
        if (w.base_index < 0) return fail(GNS_ERR_INVALID, "negative base_index");
        if (std::min(w.rows, w.cols) > kDion3MaxSelect)
            return fail(GNS_ERR_UNSUPPORTED, "selection dimension above " + std::to_string(kDion3MaxSelect));
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DeviceState* st = nullptr;
    RET(get_state(&st));
    begin_call(*st);
    std::vector<std::pair<std::pair<int, int>, std::vector<int>>> buckets;
    for (int i = 0; i < n; ++i) {
        auto key = std::make_pair(params[i].rows, params[i].cols);
        auto it = std::find_if(buckets.begin(), buckets.end(), [&](const auto& b) { return b.first == key; });
        if (it == buckets.end()) {
            buckets.push_back({key, {i}});
        } else {
            it->second.push_back(i);
        }
    }
    Coeffs cf;
    RET(load_coeffs(nullptr, 5, cf));
    for (auto& bk : buckets) {
        const int R = bk.first.first, C = bk.first.second;
        const int G = static_cast<int>(bk.second.size());
        const bool cols = R > C;  // select along the smaller dimension
        const int nsel = cols ? C : R, m = cols ? R : C;
        const int k = dion3_selection_count(nsel, fraction);
        const BucketGeom g = make_geom(k, m);
        const float scale = 0.2f * std::sqrt(static_cast<float>(std::max(R, C)));
        // Per matrix: 3 pointers, a base, the norms, the selection, the
        // positions and the gathered fp32 submatrix, all in the metadata block.
        const size_t per_meta = 3 * sizeof(void*) + sizeof(long long) + 8 * static_cast<size_t>(nsel) +
                                4 * static_cast<size_t>(k) + 4 * static_cast<size_t>(k) * m + 1024;
        int Gc = std::min(G, 65535);
        while (Gc > 1 &&
               make_layout(g, Gc, false, true, static_cast<size_t>(Gc) * per_meta).total > chunk_cap_bytes())
            Gc = (Gc + 1) / 2;
        const Layout L = make_layout(g, Gc, false, true, static_cast<size_t>(Gc) * per_meta);
        RET(ensure_workspace(*st, L.total));
        const long long ld_o = round_up_ll(m, 8);
        for (int g0 = 0; g0 < G; g0 += Gc) {
            const int gc = std::min(Gc, G - g0);
            std::vector<const void*> ptrs(3 * static_cast<size_t>(gc));
            std::vector<long long> bases(gc);
            for (int j = 0; j < gc; ++j) {
                const int i = bk.second[g0 + j];
                ptrs[j] = momentum[i].data;
                ptrs[gc + j] = grads[i].data;
                ptrs[2 * gc + j] = params[i].data;
                bases[j] = params[i].base_index;
            }
            char* meta = st->ws + L.meta;
            size_t off = 0;
            auto carve = [&](size_t bytes) {
                char* p = meta + off;
                off = align_up(off + bytes, 256);
                return p;
            };
            char* ptr_block = carve(ptrs.size() * sizeof(void*));
            long long* bases_dev = reinterpret_cast<long long*>(carve(bases.size() * sizeof(long long)));
            float* l1 = reinterpret_cast<float*>(carve(sizeof(float) * static_cast<size_t>(gc) * nsel));
            int* sel = reinterpret_cast<int*>(carve(sizeof(int) * static_cast<size_t>(gc) * k));
            int* pos = reinterpret_cast<int*>(carve(sizeof(int) * static_cast<size_t>(gc) * nsel));
            float* X = reinterpret_cast<float*>(carve(sizeof(float) * static_cast<size_t>(gc) * k * m));
            CK(cudaMemcpyAsync(ptr_block, ptrs.data(), ptrs.size() * sizeof(void*), cudaMemcpyHostToDevice, s));
            CK(cudaMemcpyAsync(bases_dev, bases.data(), bases.size() * sizeof(long long), cudaMemcpyHostToDevice, s));
            const void* const* pm = reinterpret_cast<const void* const*>(ptr_block);
            MatrixSet Ms{nullptr, 0, pm};
            MatrixSet Gs{nullptr, 0, pm + gc};
            MatrixSet Ws{nullptr, 0, pm + 2 * gc};
            LAUNCH(kClsMuon, launch_dion3_accumulate(Ms, Gs, gc, R, C, cols, l1, s));
            LAUNCH(kClsMuon, launch_dion3_select(l1, gc, nsel, k, sel, pos, s));
            LAUNCH(kClsMuon, launch_dion3_gather(Ms, gc, R, C, cols, sel, k, X, s));
            OutSpec os;
            os.out.p = st->ws + L.o16;
            os.out.rows = k;
            os.out.cols = m;
            os.out.ld = ld_o;
            os.out.stride = static_cast<long long>(k) * ld_o;
            os.out.f32 = false;
            const MatrixSet Xs{X, static_cast<long long>(k) * m, nullptr};
            RET(run_core(*st, g, L, gc, Xs, nullptr, 0.0f, 5, periodic_restarts(5, 2), cf, os, s));
            LAUNCH(kClsMuon, launch_dion3_update(Ws, Ms, os.out.p, ld_o, os.out.stride, pos, nsel, bases_dev, gc, R, C,
                                                 cols, lr, wd, scale, mu, seed, step, s));
        }
    }
    return GNS_OK;
}
}  // namespace
}  // namespace gns

using namespace gns;

extern "C" {

int gns_orthogonalize_batched(float* ptr, int G, int R, int C, int steps, int restart_at, const float* coeffs,
                              void* stream) {
    if (steps < 1 || steps > GNS_MAX_STEPS) return fail(GNS_ERR_INVALID, "steps must be in 1..GNS_MAX_STEPS");
    return orthogonalize_device(ptr, G, R, C, steps, periodic_restarts(steps, restart_at), coeffs,
                                static_cast<cudaStream_t>(stream));
}

int gns_orthogonalize_batched_schedule(float* ptr, int G, int R, int C, int steps, uint64_t restart_mask,
                                       const float* coeffs, void* stream) {
    if (steps < 1 || steps > GNS_MAX_STEPS) return fail(GNS_ERR_INVALID, "steps must be in 1..GNS_MAX_STEPS");
    const uint64_t valid = (steps >= 64 ? ~uint64_t(0) : ((uint64_t(1) << steps) - 1)) & ~uint64_t(1);
    if (restart_mask & ~valid) return fail(GNS_ERR_INVALID, "restart mask bits must lie in 1..steps-1");
    return orthogonalize_device(ptr, G, R, C, steps, restart_mask, coeffs, static_cast<cudaStream_t>(stream));
}

int gns_gram_ns_state(float* ptr, int G, int R, int C, int steps, uint64_t restart_mask, uint16_t* r_state,
                      uint16_t* q_state, float* r_scale, void* stream) {
    RET(validate_common(G, R, C, steps));
    if (G == 0) return GNS_OK;
    if (!ptr || !r_state || !q_state || !r_scale) return fail(GNS_ERR_INVALID, "null pointer");
    if (R == C) return fail(GNS_ERR_INVALID, "square matrices run standard Newton-Schulz: no Gram state");
    const uint64_t valid = (steps >= 64 ? ~uint64_t(0) : ((uint64_t(1) << steps) - 1)) & ~uint64_t(1);
    if (restart_mask & ~valid) return fail(GNS_ERR_INVALID, "restart mask bits must lie in 1..steps-1");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DeviceState* st = nullptr;
    RET(get_state(&st));
    begin_call(*st);
    Coeffs cf;
    RET(load_coeffs(nullptr, steps, cf));
    const BucketGeom g = make_geom(R, C);
    const bool direct_out = (reinterpret_cast<uintptr_t>(ptr) % 16 == 0) && ((static_cast<long long>(C) * 4) % 16 == 0);
    if (chunk_size(g, G, !direct_out, false) < G) return fail(GNS_ERR_INVALID, "bucket larger than one workspace chunk");
    const Layout L = make_layout(g, G, !direct_out, false, 0);
    RET(ensure_workspace(*st, L.total));
    const long long numel = static_cast<long long>(R) * C;
    MatrixSet in{ptr, numel, nullptr};
    OutSpec os;
    os.out.p = direct_out ? static_cast<void*>(ptr) : static_cast<void*>(st->ws + L.out32);
    os.out.rows = R;
    os.out.cols = C;
    os.out.ld = direct_out ? C : L.ld_out32;
    os.out.stride = static_cast<long long>(R) * os.out.ld;
    os.out.f32 = true;
    GramState gs;
    RET(run_core(*st, g, L, G, in, nullptr, 0.0f, steps, restart_mask, cf, os, s, &gs));
    if (!direct_out)
        LAUNCH(kClsCopy, launch_copy_rows_f32(static_cast<float*>(os.out.p), os.out.ld, os.out.stride, ptr, G, R, C, s));
    // The matrices of each state are contiguous (stride = n ld), so one 2D
    // copy per state moves G n rows of n halves.
    const int n = g.n;
    CK(cudaMemcpy2DAsync(r_state, static_cast<size_t>(n) * 2, gs.r, static_cast<size_t>(gs.ld) * 2,
                         static_cast<size_t>(n) * 2, static_cast<size_t>(G) * n, cudaMemcpyDeviceToDevice, s));
    CK(cudaMemcpy2DAsync(q_state, static_cast<size_t>(n) * 2, gs.q, static_cast<size_t>(gs.ld) * 2,
                         static_cast<size_t>(n) * 2, static_cast<size_t>(G) * n, cudaMemcpyDeviceToDevice, s));
    *r_scale = gs.s;
    return GNS_OK;
}

int gns_orthogonalize_batched_host(float* host_ptr, int G, int R, int C, int steps, int restart_at,
                                   const float* coeffs, void* stream) {
    RET(validate_common(G, R, C, steps));
    if (G == 0) return GNS_OK;
    if (!host_ptr) return fail(GNS_ERR_INVALID, "host_ptr is null");
    DeviceState* st = nullptr;
    RET(get_state(&st));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t bytes = static_cast<size_t>(G) * R * C * sizeof(float);
    if (st->stage_bytes < bytes) {
        if (st->stage) {
            CK(cudaDeviceSynchronize());
            CK(cudaFree(st->stage));
            st->stage = nullptr;
            st->stage_bytes = 0;
        }
        if (cudaMalloc(&st->stage, bytes) != cudaSuccess) {
            cudaGetLastError();
            return fail(GNS_ERR_NOMEM, "staging allocation failed");
        }
        st->stage_bytes = bytes;
    }
    if (steps < 1 || steps > GNS_MAX_STEPS) return fail(GNS_ERR_INVALID, "steps must be in 1..GNS_MAX_STEPS");
    if (!st->h2d) CK(cudaStreamCreateWithFlags(&st->h2d, cudaStreamNonBlocking));
    if (!st->d2h) CK(cudaStreamCreateWithFlags(&st->d2h, cudaStreamNonBlocking));
    // Pipelined in chunks of about 64 MiB: chunk c's host-to-device copy (one
    // copy stream), its orthogonalization (the caller's stream) and its
    // device-to-host copy (the other copy stream) overlap with the
    // neighbouring chunks' stages; events order the three stages of a chunk.
    const long long per = static_cast<long long>(R) * C;
    long long chunk_bytes = 64LL << 20;
    if (const char* e = std::getenv("GNS_HOST_CHUNK_MB")) {
        if (std::atoll(e) > 0) chunk_bytes = std::atoll(e) << 20;
    }
    const int gc = static_cast<int>(std::max(1LL, std::min<long long>(G, chunk_bytes / (per * 4))));
    // The first chunk's copy in and the last chunk's orthogonalization and
    // copy out overlap nothing, so the ends taper: a quarter chunk, then the
    // rest of a chunk, full chunks (a partial one in the middle), the rest of
    // a chunk and a quarter chunk. The link (not the GPU) bounds the middle.
    // GNS_HOST_SIZES (comma-separated matrices per chunk, summing to G)
    // overrides the schedule (tuning).
    std::vector<int> sizes;
    if (const char* e = std::getenv("GNS_HOST_SIZES")) {
        long long sum = 0;
        for (const char* q = e; *q;) {
            const long long v = std::atoll(q);
            if (v <= 0) break;
            sizes.push_back(static_cast<int>(v));
            sum += v;
            while (*q && *q != ',') ++q;
            if (*q == ',') ++q;
        }
        if (sum != G) sizes.clear();
    }
    if (sizes.empty()) {
        auto fill = [&](int rem) {
            while (rem > 0) {
                const int n = std::min(gc, rem);
                sizes.push_back(n);
                rem -= n;
            }
        };
        if (G >= 2 * gc && gc > 1) {
            const int h = std::max(1, gc / 4);
            sizes.push_back(h);
            sizes.push_back(gc - h);
            fill(G - 2 * gc);
            sizes.push_back(gc - h);
            sizes.push_back(h);
        } else {
            fill(G);
        }
    }
    const int nchunks = static_cast<int>(sizes.size());
    std::vector<cudaEvent_t> ev(2 * static_cast<size_t>(nchunks) + 1, nullptr);
    int rc = GNS_OK;
    auto cleanup = [&]() {
        for (cudaEvent_t e : ev)
            if (e) cudaEventDestroy(e);
    };
    for (cudaEvent_t& e : ev) {
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
            cudaGetLastError();
            cleanup();
            return fail(GNS_ERR_CUDA, "event creation failed");
        }
    }
    const uint64_t restarts = periodic_restarts(steps, restart_at);
    auto run = [&]() -> int {
        // The copies start after the caller's earlier work on its stream.
        CK(cudaEventRecord(ev[0], s));
        CK(cudaStreamWaitEvent(st->h2d, ev[0], 0));
        int g0 = 0;
        for (int c = 0; c < nchunks; g0 += sizes[c], ++c) {
            const int n = sizes[c];
            float* dev = st->stage + static_cast<long long>(g0) * per;
            float* host = host_ptr + static_cast<long long>(g0) * per;
            const size_t b = static_cast<size_t>(n) * per * sizeof(float);
            CK(cudaMemcpyAsync(dev, host, b, cudaMemcpyHostToDevice, st->h2d));
            CK(cudaEventRecord(ev[1 + 2 * c], st->h2d));
            CK(cudaStreamWaitEvent(s, ev[1 + 2 * c], 0));
            RET(orthogonalize_device(dev, n, R, C, steps, restarts, coeffs, s));
            CK(cudaEventRecord(ev[2 + 2 * c], s));
            CK(cudaStreamWaitEvent(st->d2h, ev[2 + 2 * c], 0));
            CK(cudaMemcpyAsync(host, dev, b, cudaMemcpyDeviceToHost, st->d2h));
        }
        CK(cudaStreamSynchronize(st->d2h));
        CK(cudaStreamSynchronize(s));
        return GNS_OK;
    };
    rc = run();
    if (rc != GNS_OK) {
        cudaStreamSynchronize(st->h2d);
        cudaStreamSynchronize(st->d2h);
        cudaStreamSynchronize(s);
    }
    cleanup();
    return rc;
}

int muon_step(const gns_tensor* params, const gns_tensor* grads, const gns_tensor* momentum, int n, float lr,
              float wd, float mu, uint64_t seed, uint64_t step, void* stream) {
    return optimizer_step(params, grads, momentum, nullptr, n, lr, wd, mu, 0.0f, 0.0f, seed, step, stream);
}

int dion3_step(const gns_tensor* params, const gns_tensor* grads, const gns_tensor* momentum, int n,
               float fraction, float lr, float wd, float mu, uint64_t seed, uint64_t step, void* stream) {
    return dion3_step_impl(params, grads, momentum, n, fraction, lr, wd, mu, seed, step, stream);
}

int normuon_step(const gns_tensor* params, const gns_tensor* grads, const gns_tensor* momentum,
                 const gns_tensor* second_moments, int n, float lr, float wd, float mu, float beta2, float eps,
                 uint64_t seed, uint64_t step, void* stream) {
    if (n > 0 && !second_moments) return fail(GNS_ERR_INVALID, "null second-moment array");
    return optimizer_step(params, grads, momentum, second_moments, n, lr, wd, mu, beta2, eps, seed, step, stream);
}

int gns_muon_momentum(float* M, const uint16_t* G_bf16, int64_t numel, float mu, void* stream) {
    if (numel < 0 || (numel > 0 && (!M || !G_bf16))) return fail(GNS_ERR_INVALID, "bad momentum arguments");
    if (numel == 0) return GNS_OK;
    DeviceState* st = nullptr;
    RET(get_state(&st));
    MatrixSet Ms{M, numel, nullptr};
    MatrixSet Gs{G_bf16, numel, nullptr};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    LAUNCH(kClsMuon, launch_momentum(Ms, Gs, numel, 1, mu, s));
    return GNS_OK;
}

int gns_muon_update(uint16_t* W_bf16, const uint16_t* O_fp16, int rows, int cols, float lr, float wd, float scale,
                    uint64_t seed, uint64_t step, int64_t base_index, void* stream) {
    if (rows < 0 || cols < 0 || base_index < 0) return fail(GNS_ERR_INVALID, "bad update arguments");
    if (static_cast<long long>(rows) * cols == 0) return GNS_OK;
    if (!W_bf16 || !O_fp16) return fail(GNS_ERR_INVALID, "null pointer");
    DeviceState* st = nullptr;
    RET(get_state(&st));
    const long long numel = static_cast<long long>(rows) * cols;
    MatrixSet Ws{W_bf16, numel, nullptr};
    MatrixSet Os{O_fp16, numel, nullptr};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    LAUNCH(kClsMuon, launch_muon_update(Ws, Os, cols, nullptr, base_index, 1, rows, cols, lr, wd, scale, seed, step,
                                        st->num_sms, s));
    return GNS_OK;
}

int gns_symm_gemm(const void* A, const void* B, const void* C, void* D, int G, int n, int k, float alpha, float beta,
                  void* stream) {
    if (G < 0 || n < 1 || k < 1) return fail(GNS_ERR_INVALID, "G >= 0, n >= 1 and k >= 1 required");
    if (G == 0) return GNS_OK;
    if (!A || !B || !D) return fail(GNS_ERR_INVALID, "null pointer");
    if (n % 8 || k % 8) return fail(GNS_ERR_INVALID, "n and k must be multiples of 8");
    for (const void* q : {A, B, C, static_cast<const void*>(D)})
        if (reinterpret_cast<uintptr_t>(q) % 16 != 0) return fail(GNS_ERR_INVALID, "pointers must be 16-byte aligned");
    DeviceState* st = nullptr;
    RET(get_state(&st));
    begin_call(*st);
    Mat a{const_cast<void*>(A), n, k, k, static_cast<long long>(n) * k, false};
    Mat b{const_cast<void*>(B), n, k, k, static_cast<long long>(n) * k, false};
    Mat d{D, n, n, n, static_cast<long long>(n) * n, false};
    Mat c{const_cast<void*>(C), n, n, n, static_cast<long long>(n) * n, false};
    ProblemSpec p;
    p.A = a;
    p.B = b;
    p.D = d;
    p.Dt = &d;
    p.C = C ? &c : nullptr;
    p.alpha = alpha;
    p.beta = C ? beta : 0.0f;
    p.sym = true;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const TileShape ts = choose_tile(n, G, st->num_sms);
    RET(ensure_workspace(*st, 256));
    ProgramBuilder prog(*st, G, ts, reinterpret_cast<int*>(st->ws), s);
    RET(prog.phase(p, nullptr));
    return prog.flush();
}

int gns_get_status(void* stream) {
    int dev = 0;
    CK(cudaGetDevice(&dev));
    CK(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    // The status words of this device: the allocating entry points' and the
    // allocation-free entry point's (inside its fixed array). Neither is
    // created here, so this call allocates nothing.
    int* words[2] = {nullptr, nullptr};
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = g_dev.find(dev);
        if (it != g_dev.end()) words[0] = it->second.err;
    }
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        auto it = g_noalloc.find(dev);
        if (it != g_noalloc.end() && it->second.ready) words[1] = reinterpret_cast<int*>(it->second.scratch);
    }
    int result = GNS_OK;
    for (int* w : words) {
        if (!w) continue;
        int v = 0;
        CK(cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost));
        if (v != 0) {
            CK(cudaMemset(w, 0, sizeof(int)));
            if (result == GNS_OK) result = v;
        }
    }
    return result;
}

int gns_test_bounded_wait(int kind, int64_t limit_ns, void* stream) {
    if (kind < 0 || kind > 1) return fail(GNS_ERR_INVALID, "kind must be 0 (mbarrier) or 1 (counter)");
    if (limit_ns < 1000 || limit_ns > 1000000000LL) return fail(GNS_ERR_INVALID, "limit_ns must be in [1 us, 1 s]");
    DeviceState* st = nullptr;
    RET(get_state(&st));
    begin_call(*st);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    DevStatus first = st->status;
    first.limit_ns = static_cast<unsigned long long>(limit_ns);
    DevStatus rest = first;
    rest.limit_ns = std::min<unsigned long long>(1000ull * first.limit_ns, 10000000000ull);
    // Words 2 and 3 of the status block: a counter nothing writes (zero since
    // the block was allocated) and the count of waits that gave up.
    const int* never = st->err + 2;
    int* gave_up = st->err + 3;
    CK(cudaMemsetAsync(gave_up, 0, sizeof(int), s));
    LAUNCH(kClsMuon, launch_bounded_wait_test(first, rest, kind, never, gave_up, s));
    CK(cudaStreamSynchronize(s));
    int v = 0;
    CK(cudaMemcpy(&v, gave_up, sizeof(int), cudaMemcpyDeviceToHost));
    return v;
}

const char* gns_status_string(int status) {
    switch (status) {
        case GNS_OK: return "ok";
        case GNS_ERR_INVALID: return "invalid argument";
        case GNS_ERR_CUDA: return "CUDA runtime error";
        case GNS_ERR_NONFINITE: return "non-finite input norm";
        case GNS_ERR_TIMEOUT: return "device wait timed out";
        case GNS_ERR_NOMEM: return "out of device memory";
        case GNS_ERR_UNSUPPORTED: return "unsupported device (sm_103a required)";
        default: return "unknown status";
    }
}

const char* gns_last_error(void) { return g_last_error.c_str(); }

int64_t gns_launch_count(void) { return g_launches.load(); }

void gns_profile_enable(int on) { g_profiling.store(on != 0); }

int gns_profile_read(int64_t* counts, double* ms, int max_classes) {
    std::vector<ProfRec> recs;
    {
        std::lock_guard<std::mutex> lk(g_prof_mu);
        recs.swap(g_recs);
    }
    std::vector<int64_t> c(kNumCls, 0);
    std::vector<double> t(kNumCls, 0.0);
    int rc = GNS_OK;
    for (auto& r : recs) {
        float e = 0.0f;
        cudaError_t err = cudaEventSynchronize(r.b);
        if (err == cudaSuccess) err = cudaEventElapsedTime(&e, r.a, r.b);
        if (err != cudaSuccess) {
            rc = cuda_fail(err, "cudaEventElapsedTime");
        } else {
            c[r.cls] += 1;
            t[r.cls] += e;
        }
    }
    {
        std::lock_guard<std::mutex> lk(g_prof_mu);
        for (auto& r : recs) {
            g_event_pool.push_back(r.a);
            g_event_pool.push_back(r.b);
        }
    }
    for (int k = 0; k < kNumCls && k < max_classes; ++k) {
        if (counts) counts[k] = c[k];
        if (ms) ms[k] = t[k];
    }
    return rc == GNS_OK ? kNumCls : rc;
}

int64_t gns_workspace_bytes(void) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_dev.find(dev);
    return it == g_dev.end() ? 0 : static_cast<int64_t>(it->second.ws_bytes);
}

void gns_release(void) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_dev.find(dev);
    if (it == g_dev.end()) return;
    cudaDeviceSynchronize();
    if (it->second.ws) cudaFree(it->second.ws);
    if (it->second.stage) cudaFree(it->second.stage);
    it->second.ws = nullptr;
    it->second.ws_bytes = 0;
    it->second.stage = nullptr;
    it->second.stage_bytes = 0;
    if (it->second.h2d) cudaStreamDestroy(it->second.h2d);
    if (it->second.d2h) cudaStreamDestroy(it->second.d2h);
    it->second.h2d = it->second.d2h = nullptr;
}

}  // extern "C"

extern "C" int gns_orthogonalize_batched_noalloc(float* ptr, int G, int R, int C, int steps, int restart_at,
                                                 const float* coeffs, void* stream) {
    RET(validate_common(G, R, C, steps));
    if (G == 0) return GNS_OK;
    if (!ptr) return fail(GNS_ERR_INVALID, "ptr is null");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    CK(cudaGetDevice(&dev));
    NoAllocDevice nd;
    {
        // First call on a device: look up the array's device address (the
        // name is only a host-side stand-in) and the SM count. No allocation.
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        NoAllocDevice& e = g_noalloc[dev];
        if (!e.ready) {
            CK(cudaDeviceGetAttribute(&e.num_sms, cudaDevAttrMultiProcessorCount, dev));
            // The same SM cap as the allocating entry points (GNS_NUM_SMS).
            const char* cap = std::getenv("GNS_NUM_SMS");
            if (cap && std::atoi(cap) > 0) e.num_sms = std::min(e.num_sms, std::atoi(cap));
            CK(cudaDeviceGetAttribute(&e.cc_major, cudaDevAttrComputeCapabilityMajor, dev));
            CK(cudaDeviceGetAttribute(&e.cc_minor, cudaDevAttrComputeCapabilityMinor, dev));
            void* addr = nullptr;
            CK(cudaGetSymbolAddress(&addr, g_noalloc_scratch));
            e.scratch = static_cast<char*>(addr);
            e.ready = true;
        }
        e.epoch = e.epoch == 0x7fffffff ? 1 : e.epoch + 1;
        nd = e;
    }
    if (!(nd.cc_major == 10 && nd.cc_minor == 3))
        return fail(GNS_ERR_UNSUPPORTED, "this library is built for sm_103a (GB300) only");
    Coeffs cf;
    RET(load_coeffs(coeffs, steps, cf));
    const BucketGeom g = make_geom(R, C);
    const bool direct_out = (reinterpret_cast<uintptr_t>(ptr) % 16 == 0) && ((static_cast<long long>(C) * 4) % 16 == 0);
    // Largest chunk of matrices whose workspace fits in the fixed array.
    const size_t avail = kNoAllocBytes - kNoAllocStatusBytes;
    const size_t per = make_layout(g, 1, !direct_out, false, 0).total;
    if (per > avail)
        return fail(GNS_ERR_INVALID, "a " + std::to_string(R) + " x " + std::to_string(C) + " matrix needs " +
                                         std::to_string(per) + " bytes of workspace; the allocation-free entry point has " +
                                         std::to_string(avail) + " bytes");
    int Gc = static_cast<int>(std::min<size_t>(std::min<size_t>(G, 65535), avail / per));
    while (Gc > 1 && make_layout(g, Gc, !direct_out, false, 0).total > avail) --Gc;
    const Layout L = make_layout(g, Gc, !direct_out, false, 0);

    DeviceState st;
    st.device = dev;
    st.num_sms = nd.num_sms;
    st.cc_major = nd.cc_major;
    st.cc_minor = nd.cc_minor;
    st.err = reinterpret_cast<int*>(nd.scratch);
    st.epoch = nd.epoch;
    st.status = DevStatus{st.err, st.epoch, 0, wait_limit_ns()};
    st.ws = nd.scratch + kNoAllocStatusBytes;
    st.ws_bytes = avail;
    // The array keeps the previous call's contents. The status word starts at
    // zero (the array is zero when the library loads) and is cleared by
    // gns_get_status; the abort mark holds an earlier call's number, which no
    // later call's waits take for their own; every workspace byte a kernel
    // reads is written first in the same call (the counters by the
    // stream-ordered clear before each GEMM launch).

    const long long numel = static_cast<long long>(R) * C;
    for (int g0 = 0; g0 < G; g0 += Gc) {
        const int gc = std::min(Gc, G - g0);
        float* base = ptr + static_cast<long long>(g0) * numel;
        MatrixSet in{base, numel, nullptr};
        OutSpec os;
        os.out.rows = R;
        os.out.cols = C;
        os.out.f32 = true;
        if (direct_out) {
            os.out.p = base;
            os.out.ld = C;
            os.out.stride = numel;
        } else {
            os.out.p = st.ws + L.out32;
            os.out.ld = L.ld_out32;
            os.out.stride = static_cast<long long>(R) * L.ld_out32;
        }
        RET(run_core(st, g, L, gc, in, nullptr, 0.0f, steps, periodic_restarts(steps, restart_at), cf, os, s));
        if (!direct_out)
            LAUNCH(kClsCopy, launch_copy_rows_f32(static_cast<float*>(os.out.p), os.out.ld, os.out.stride, base, gc, R, C, s));
    }
    return GNS_OK;
}
