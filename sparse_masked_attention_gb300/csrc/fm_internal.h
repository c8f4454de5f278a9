// fm_internal.h -- host-side structures shared by the library's translation
// units: problem geometry, the workspace layout and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "flashmask.h"

namespace fm {

constexpr int TILE = 128;  // tile edge of the tile map and of the list entries

// Error codes a kernel may leave in its device error word (bits).
enum : unsigned { ERR_NONE = 0, ERR_TIMEOUT = 1, ERR_SMEM_ALIGN = 2, ERR_BOUNDS = 4 };

struct Geometry {
    int B, H, Hm, N, d, dv;
    int T;       // ceil(N / 128)
    int Npad;    // T * 128
    float scale;
    int causal;
    uint64_t timeout_ns;
    int deterministic;
    const float *sink;  // [H] attention-sink logits, or nullptr
    float *dsink;       // [H] their gradient (backward), or nullptr
    int reuse_map;      // the workspace already holds this problem's tile map and lists
    int debug_bounds;   // attention kernels check their work lists before use
    int acc32;          // backward: add the gradients to fp32 outputs instead of writing bf16
    int drop_load;      // failure-detection test: the forward skips one K load (0: off)
};

// Normalised mask boundaries per key column: (LTS, LTE, UTS, UTE) clamped to
// [0, N]; absent intervals empty; padding columns j >= N masked for every row.
struct Workspace {
    int4 *vec;         // [B*Hm][Npad]
    uint8_t *cls;      // [B*Hm][T][T] tile classes
    int *fwd_list;     // [B*Hm][T][T] per q-tile: (kt << 1) | needs_mask
    int *fwd_cnt;      // [B*Hm][T]
    int *bwd_list;     // [B*Hm][T][T] per k-tile: (qt << 1) | needs_mask
    int *bwd_cnt;      // [B*Hm][T]
    int *pair_list;    // [B*Hm][TP][T] per pair of q-tiles (2p, 2p+1), TP = ceil(T/2):
                       // (kt << 2) | (needs_mask of 2p) << 1 | needs_mask of 2p+1,
                       // every k-tile either q-tile keeps; a tile one of them skips
                       // counts as needing the mask for it
    int *pair_cnt;     // [B*Hm][TP]
    int *pair_order;   // [B*Hm][TP] pair indices by decreasing key-tile count
    float *lse2;       // [B*H][Npad] log2-domain LSE, +inf for empty / padding rows
    float *delta;      // [B*H][Npad] D_i = sum_c dO_ic O_ic
    void *v16;         // [B,N,H,dv] fp16 copy of V * s_v   (backward)
    void *do16;        // [B,N,H,dv] fp16 copy of dO * s_o  (backward)
    float *sink_part;  // [B*H*Npad/16] per-block sink-gradient sums (backward)
    uint2 *range_part; // [B*H][T] largest |dO| and |V| (bf16 bit patterns) per row tile
    float4 *scales;    // [B*H] (s_o, s_v, 1/s_o, 1/(s_o s_v)): powers of two that put the
                       // largest |dO| and |V| of the (batch, head) in [2^14, 2^15)
    float4 *dqacc;     // fused backward: fp32 dQ sums [B*H][d/4][Npad] (float4)
};

// SMs of the current device: with one resident CTA per SM, a kernel's next
// wave starts this many blocks later.  0 when it cannot be read.
inline int current_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return 0;
    return sms;
}

// The backward reduces dQ inside its key-side kernel (one pass, fp32 red.add
// into Workspace::dqacc) at d = dv <= 128 unless the deterministic mode asks
// for the atomic-free split (key side, then query side).
inline bool fused_dq(const Geometry &g) {
    return !g.deterministic && g.d == g.dv && g.d <= 128;
}

// Optional per-kernel event recording (fm_options.kernel_events).
struct Recorder {
    cudaEvent_t *ev = nullptr;
    int n = 0;
    int i = 0;
    void before(cudaStream_t s) {
        if (ev && 2 * i + 1 < n) cudaEventRecord(ev[2 * i], s);
    }
    void after(cudaStream_t s) {
        if (ev && 2 * i + 1 < n) cudaEventRecord(ev[2 * i + 1], s);
        ++i;
    }
};

// Launches `kern` with programmatic stream serialization: its CTAs may start
// while the previous kernel in the stream drains.  Every kernel launched this
// way calls pdl_wait() before it touches memory an earlier kernel in the
// stream may write or read, so the stream order of all results is that of
// plain launches.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// Text returned by flashmask_last_error_detail on this thread (api.cu).
void set_error_detail(const char *msg);
// Makes the device that owns `anchor` (device memory) current for this
// thread and checks that it is an sm_103 part (api.cu).
bool bind_device(const void *anchor);

// Keeps the calling thread's CUDA context: records the current context when
// an entry point starts and makes it current again when the entry point
// returns.  Entry points make the device of the caller's memory current for
// their own launches; with this guard the caller finds its thread as it left
// it (api.cu).
class CallerContext {
  public:
    CallerContext();
    ~CallerContext();
    CallerContext(const CallerContext &) = delete;
    CallerContext &operator=(const CallerContext &) = delete;

  private:
    CUcontext saved_ = nullptr;
    bool valid_ = false;
};

// Lays the workspace out from `base` (may be nullptr to size it); returns bytes.
size_t carve_workspace(const Geometry &g, bool bwd, void *base, Workspace *ws);

struct MaskPtrs {
    const int32_t *lts, *lte, *uts, *ute;
};

// classify.cu
cudaError_t launch_classify(const Geometry &g, const MaskPtrs &m, const Workspace &ws,
                            cudaStream_t st);
cudaError_t launch_fwd_lists(const Geometry &g, const Workspace &ws, cudaStream_t st);
// debug_bounds: checks (and neutralises) every work list in the workspace.
cudaError_t launch_validate_lists(const Geometry &g, const Workspace &ws, cudaStream_t st);
// A bounded wait that nothing completes (failure-detection self-test).
cudaError_t launch_wait_selftest(uint64_t timeout_ns, cudaStream_t st);
cudaError_t launch_count(const Geometry &g, const MaskPtrs &m, unsigned long long *counts,
                         cudaStream_t st);
unsigned read_clear_error_classify();

// fwd.cu
// Box heights (rows) of the K/V tensor maps the forward kernel expects.
int fwd_key_rows(int d, int dv);

struct FwdArgs {
    const CUtensorMap *tm_q, *tm_k, *tm_v;
    int k_rows;  // box height of tm_k / tm_v; must equal the kernel's key tile
    const CUtensorMap *tm_o;  // O, 64-column x 128-row boxes (the output is stored by TMA)
    void *o;
    float *lse;
};
cudaError_t launch_fwd(const Geometry &g, const Workspace &ws, const FwdArgs &a,
                       cudaStream_t st);
unsigned read_clear_error_fwd();

// bwd.cu
// Box heights the backward kernels expect: key sub-tile of the query-side
// kernel (its K/V maps) and query sub-tile of the key-side kernel (its Q/dO maps).
int dq_key_rows(int d, int dv);
int dkdv_query_rows(int d, int dv);

struct BwdArgs {
    int dq_k_rows;   // box height of tm_k_dq / tm_v_dq
    int kv_q_rows;   // box height of tm_q / tm_do
    // key-side (dK/dV) kernel maps: q/dO boxes of its query sub-tile, k/v of 128 rows
    const CUtensorMap *tm_q, *tm_k, *tm_v, *tm_do;
    // query-side (dQ) kernel maps: q/dO boxes of 128 rows, k/v of its key sub-tile
    const CUtensorMap *tm_q_dq, *tm_k_dq, *tm_v_dq, *tm_do_dq;
    // outputs, 64-column x 128-row boxes (stored by TMA)
    const CUtensorMap *tm_dq_out, *tm_dk_out, *tm_dv_out;
    const void *o, *v, *dout;
    const float *lse;
    void *dq, *dk, *dv;
};
cudaError_t launch_bwd(const Geometry &g, const Workspace &ws, const BwdArgs &a,
                       cudaStream_t st, Recorder &rec);
unsigned read_clear_error_bwd();

}  // namespace fm
