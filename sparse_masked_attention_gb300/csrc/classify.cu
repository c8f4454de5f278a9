// classify.cu -- the tile map: which 128x128 (query-tile, key-tile) blocks are
// fully masked (skipped), partially masked (mask applied elementwise) or
// unmasked.  This is the sparsity skipping of "FlashMask: Efficient and Rich
// Mask Extension of FlashAttention" (abstract) on the column-wise boundaries
// of the FlashMask README ("Overview").
//
// One CTA per (mask head, key tile).  Its 128 threads each own one key column.
// The CTA first reduces the per-tile min/max of the four boundary vectors.
// Those eight numbers settle most tiles at once.  A tile they leave open gets
// an exact per-column test: each column's masked rows form the union of at most
// three intervals ([0, j) for the causal flag, LT, UT).  The map is therefore
// exact, never just conservative.
//
// Also here: the list builder (fwd_lists_kernel), the unmasked-pair count
// (count_kernel), the debug_bounds check of every work list in a workspace
// (validate_lists_kernel) and the bounded-wait self-test
// (wait_selftest_kernel).
#include <cuda_runtime.h>
#include <stdint.h>

#include "fm_device.cuh"
#include "fm_internal.h"

namespace fm {

static __device__ unsigned g_err_classify;

namespace {

__device__ __forceinline__ int clampN(int x, int N) { return x < 0 ? 0 : (x > N ? N : x); }

// Does [a, b) meet [r0, r1)?
__device__ __forceinline__ bool meets(int a, int b, int r0, int r1) {
    return max(a, r0) < min(b, r1);
}

// Does the union of [0, cj) (cj = j under the causal flag, else 0),
// [c.x, c.y) and [c.z, c.w) cover [r0, r1)?
__device__ __forceinline__ bool covers(int cj, int4 c, int r0, int r1) {
    int reach = r0;
#pragma unroll
    for (int round = 0; round < 3; ++round) {
        if (0 <= reach && cj > reach) reach = cj;
        if (c.x <= reach && c.y > reach) reach = c.y;
        if (c.z <= reach && c.w > reach) reach = c.w;
    }
    return reach >= r1;
}

constexpr int kClassifyChunk = 32;  // most query tiles per classify CTA

__device__ __forceinline__ int warp_min(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// One CTA per (key tile, chunk of at most kClassifyChunk query tiles, mask head).
// Per query tile qt, one word of `state` collects the CTA's decision:
//   bits 0..3  column test "every column of warp w covers the tile"
//   bits 4..7  column test "some column of warp w reaches into the tile"
//   bit  8     the column test ran (the tile map's min/max left the tile open)
//   bits 9..10 the class + 1, when the min/max settled the tile
// The loop over query tiles needs no CTA barrier: warps vote on their own and
// OR their bits in; after one barrier the classes are written.
__global__ void __launch_bounds__(128) classify_kernel(
    int N, int T, int Npad, int Hm, int causal, int chunk, const int32_t *__restrict__ lts,
    const int32_t *__restrict__ lte, const int32_t *__restrict__ uts,
    const int32_t *__restrict__ ute, int4 *__restrict__ vec, uint8_t *__restrict__ cls) {
    __shared__ unsigned state[kClassifyChunk];
    __shared__ int red[4][8];
    pdl_wait();  // the vectors and the workspace belong to earlier stream work
    pdl_trigger();
    const int kt = blockIdx.x;
    const int q_begin = blockIdx.y * chunk;
    const int q_end = min(T, q_begin + chunk);
    const int bm = blockIdx.z;  // b * Hm + hm
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = kt * TILE + threadIdx.x;
    const bool in_range = j < N;
    const size_t row = static_cast<size_t>(bm) * N;

    int4 c;
    if (in_range) {
        c.x = lts ? clampN(lts[row + j], N) : N;
        c.y = lte ? clampN(lte[row + j], N) : N;
        c.z = uts ? clampN(uts[row + j], N) : 0;
        c.w = ute ? clampN(ute[row + j], N) : 0;
    } else {
        c = make_int4(0, N, 0, 0);  // padding column: masked for every row
    }
    if (blockIdx.y == 0) vec[static_cast<size_t>(bm) * Npad + j] = c;
    for (int q = threadIdx.x; q < kClassifyChunk; q += 128) state[q] = 0u;

    // Per-tile min/max over in-range columns (padding columns are neutral):
    // warp reductions, then one exchange through shared memory.
    const int BIG = 0x7fffffff;
    int mm[8] = {in_range ? c.x : BIG, in_range ? -c.x : BIG, in_range ? c.y : BIG,
                 in_range ? -c.y : BIG, in_range ? c.z : BIG, in_range ? -c.z : BIG,
                 in_range ? c.w : BIG, in_range ? -c.w : BIG};
#pragma unroll
    for (int i = 0; i < 8; ++i) mm[i] = warp_min(mm[i]);
    if (lane == 0)
#pragma unroll
        for (int i = 0; i < 8; ++i) red[warp][i] = mm[i];
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; ++i) mm[i] = min(min(red[0][i], red[1][i]), min(red[2][i], red[3][i]));
    const int mn_lts = mm[0], mx_lts = -mm[1], mn_lte = mm[2], mx_lte = -mm[3];
    const int mn_uts = mm[4], mx_uts = -mm[5], mn_ute = mm[6], mx_ute = -mm[7];
    const int j_first = kt * TILE;
    const int j_last = min(kt * TILE + TILE, N) - 1;
    const int cj = causal ? j : 0;

    for (int qt = q_begin; qt < q_end; ++qt) {
        const int r0 = qt * TILE;
        const int r1 = min(r0 + TILE, N);
        // All columns covered by one mechanism alone.
        if ((causal && j_first >= r1) || (mx_lts <= r0 && mn_lte >= r1) ||
            (mx_uts <= r0 && mn_ute >= r1)) {
            if (threadIdx.x == 0) atomicOr(&state[qt - q_begin], (FM_TILE_SKIP + 1u) << 9);
        } else if ((!causal || j_last <= r0) && (mn_lts >= r1 || mx_lte <= r0) &&
                   (mn_uts >= r1 || mx_ute <= r0)) {
            // No mechanism reaches into the tile.
            if (threadIdx.x == 0) atomicOr(&state[qt - q_begin], (FM_TILE_UNMASKED + 1u) << 9);
        } else {
            const bool col_cov = !in_range || covers(cj, c, r0, r1);
            const bool col_touch = in_range && ((causal && j > r0) || meets(c.x, c.y, r0, r1) ||
                                                meets(c.z, c.w, r0, r1));
            const bool all_cov = __all_sync(0xffffffffu, col_cov);
            const bool any_touch = __any_sync(0xffffffffu, col_touch);
            if (lane == 0)
                atomicOr(&state[qt - q_begin], (all_cov ? 1u << warp : 0u) |
                                                   (any_touch ? 16u << warp : 0u) | 0x100u);
        }
    }
    __syncthreads();
    for (int qt = q_begin + threadIdx.x; qt < q_end; qt += 128) {
        const unsigned v = state[qt - q_begin];
        int klass;
        if (v & 0x100u)
            klass = (v & 0xfu) == 0xfu ? FM_TILE_SKIP
                                       : ((v & 0xf0u) ? FM_TILE_PARTIAL : FM_TILE_UNMASKED);
        else
            klass = static_cast<int>((v >> 9) & 3u) - 1;
        cls[(static_cast<size_t>(bm) * T + qt) * T + kt] = static_cast<uint8_t>(klass);
    }
}

// One launch, 1024-thread blocks, four jobs:
// - one warp per (mask head, q-tile): the ordered list of its non-skipped
//   k-tiles;
// - one warp per (mask head, k-tile): the ordered list of its non-skipped
//   q-tiles (the key-side backward);
// - one warp per (mask head, q-tile pair): the ordered union of the pair's
//   lists, with a needs-mask bit per q-tile (a tile the q-tile skips needs it
//   too);
// - one block per mask head, after the list blocks: the pairs by decreasing
//   length of that union, ties by index (the forward hands them out heaviest
//   first).  Its warps count the union lengths from the tile map themselves,
//   so the job needs no other block's output.
__global__ void __launch_bounds__(1024, 1) fwd_lists_kernel(int N, int T, int rows, int pair_rows,
                                                         int list_blocks,
                                                         const uint8_t *__restrict__ cls,
                                                         int *__restrict__ fwd_list,
                                                         int *__restrict__ fwd_cnt,
                                                         int *__restrict__ bwd_list,
                                                         int *__restrict__ bwd_cnt,
                                                         int *__restrict__ pair_list,
                                                         int *__restrict__ pair_cnt,
                                                         int *__restrict__ pair_order) {
    pdl_wait();  // the tile map of the kernel before
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int TP = (T + 1) / 2;
    if (static_cast<int>(blockIdx.x) >= list_blocks) {
        extern __shared__ int pcnt[];  // [TP]
        const int bm = blockIdx.x - list_blocks;
        for (int pp = warp; pp < TP; pp += 32) {  // a warp per pair, lanes over kt
            const uint8_t *a = cls + (static_cast<size_t>(bm) * T + 2 * pp) * T;
            const bool has_b = 2 * pp + 1 < T;
            int c = 0;
            for (int kt = lane; kt < T; kt += 32)
                c += (a[kt] != FM_TILE_SKIP || (has_b && a[T + kt] != FM_TILE_SKIP)) ? 1 : 0;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
            if (lane == 0) pcnt[pp] = c;
        }
        __syncthreads();
        for (int pp = threadIdx.x; pp < TP; pp += blockDim.x) {
            const int c = pcnt[pp];
            int rank = 0;
            for (int k = 0; k < TP; ++k) {
                const int ck = pcnt[k];
                rank += (ck > c || (ck == c && k < pp)) ? 1 : 0;
            }
            pair_order[static_cast<size_t>(bm) * TP + rank] = pp;
        }
        return;
    }
    const int r = blockIdx.x * 32 + warp;  // (bm * T + qt), then pairs
    const bool has_tail = (N % TILE) != 0;
    if (r < rows) {
        const uint8_t *src = cls + static_cast<size_t>(r) * T;
        int *dst = fwd_list + static_cast<size_t>(r) * T;
        int count = 0;
        for (int k0 = 0; k0 < T; k0 += 32) {
            const int kt = k0 + lane;
            const int c = kt < T ? src[kt] : FM_TILE_SKIP;
            const bool keep = c != FM_TILE_SKIP;
            const unsigned ballot = __ballot_sync(0xffffffffu, keep);
            if (keep) {
                const int pos = count + __popc(ballot & ((1u << lane) - 1u));
                const bool need = c == FM_TILE_PARTIAL || (has_tail && kt == T - 1);
                dst[pos] = (kt << 1) | (need ? 1 : 0);
            }
            count += __popc(ballot);
        }
        if (lane == 0) fwd_cnt[r] = count;
        return;
    }
    if (r < 2 * rows) {  // (bm * T + kt): the column kt of the map, over qt
        const int kr = r - rows;
        const int bm = kr / T, kt = kr % T;
        const uint8_t *src = cls + static_cast<size_t>(bm) * T * T + kt;
        int *dst = bwd_list + static_cast<size_t>(kr) * T;
        const bool tail_kt = has_tail && kt == T - 1;
        int count = 0;
        for (int q0 = 0; q0 < T; q0 += 32) {
            const int qt = q0 + lane;
            const int c = qt < T ? src[static_cast<size_t>(qt) * T] : FM_TILE_SKIP;
            const bool keep = c != FM_TILE_SKIP;
            const unsigned ballot = __ballot_sync(0xffffffffu, keep);
            if (keep)
                dst[count + __popc(ballot & ((1u << lane) - 1u))] =
                    (qt << 1) | ((c == FM_TILE_PARTIAL || tail_kt) ? 1 : 0);
            count += __popc(ballot);
        }
        if (lane == 0) bwd_cnt[kr] = count;
        return;
    }
    const int pr = r - 2 * rows;  // (bm * TP + p)
    if (pr >= pair_rows) return;
    const int bm = pr / TP, pp = pr % TP;
    const uint8_t *src_a = cls + (static_cast<size_t>(bm) * T + 2 * pp) * T;
    const bool has_b = 2 * pp + 1 < T;
    const uint8_t *src_b = src_a + T;
    int *dst = pair_list + static_cast<size_t>(pr) * T;
    int count = 0;
    for (int k0 = 0; k0 < T; k0 += 32) {
        const int kt = k0 + lane;
        const int ca = kt < T ? src_a[kt] : FM_TILE_SKIP;
        const int cb = (kt < T && has_b) ? src_b[kt] : FM_TILE_SKIP;
        const bool keep = ca != FM_TILE_SKIP || cb != FM_TILE_SKIP;
        const unsigned ballot = __ballot_sync(0xffffffffu, keep);
        if (keep) {
            const bool tail = has_tail && kt == T - 1;
            const bool need_a = ca != FM_TILE_UNMASKED || tail;
            const bool need_b = cb != FM_TILE_UNMASKED || tail;
            dst[count + __popc(ballot & ((1u << lane) - 1u))] =
                (kt << 2) | (need_a ? 2 : 0) | (need_b ? 1 : 0);
        }
        count += __popc(ballot);
    }
    if (lane == 0) pair_cnt[pr] = count;
}

// debug_bounds: checks every work list the attention kernels will read from
// the workspace, one warp per job, before they run.  A list row must have a
// count in [0, T] and entries whose tile index (entry >> shift) lies in
// [0, T); a pair-order entry must lie in [0, TP).  A failing row gets count 0
// and a failing order entry its own position (a valid pair index), so the
// kernels after it read nothing out of range; the error word records
// ERR_BOUNDS.  Jobs: fwd lists, bwd lists (rows x T entries, shift 1), pair
// lists (pair_rows x T, shift 2), pair order (pair_rows).
__global__ void __launch_bounds__(256) validate_lists_kernel(
    int T, int rows, int pair_rows, int *__restrict__ fwd_list, int *__restrict__ fwd_cnt,
    int *__restrict__ bwd_list, int *__restrict__ bwd_cnt, int *__restrict__ pair_list,
    int *__restrict__ pair_cnt, int *__restrict__ pair_order) {
    pdl_wait();  // the lists of the kernels before
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const long long job = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int TP = (T + 1) / 2;
    const int *list;
    int *cnt;
    int shift;
    long long r = job;
    if (r < rows) {
        list = fwd_list, cnt = fwd_cnt, shift = 1;
    } else if ((r -= rows) < rows) {
        list = bwd_list, cnt = bwd_cnt, shift = 1;
    } else if ((r -= rows) < pair_rows) {
        list = pair_list, cnt = pair_cnt, shift = 2;
    } else if ((r -= pair_rows) < pair_rows) {
        if (lane == 0) {
            const int v = pair_order[r];
            if (v < 0 || v >= TP) {
                pair_order[r] = static_cast<int>(r % TP);
                atomicOr(&g_err_classify, ERR_BOUNDS);
            }
        }
        return;
    } else {
        return;
    }
    const int n = cnt[r];
    bool ok = n >= 0 && n <= T;
    if (ok) {
        const int *row = list + r * T;
        for (int i = lane; i < n; i += 32) {
            const int t = row[i] >> shift;
            ok = ok && t >= 0 && t < T;
        }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (!ok && lane == 0) {
        cnt[r] = 0;
        atomicOr(&g_err_classify, ERR_BOUNDS);
    }
}

// Failure-detection self-test: one thread waits, with the caller's limit, on
// the first phase of an mbarrier that nothing arrives at.  The bounded wait
// gives up and records ERR_TIMEOUT in the error word, as the wait of any
// kernel of the library would; the kernel then returns normally.
__global__ void __launch_bounds__(32) wait_selftest_kernel(uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort = 0;
        fence_barrier_init();
        (void)mbar_wait(&bar, 0, timeout_ns, reinterpret_cast<volatile int *>(&abort),
                        &g_err_classify);
    }
}

// Unmasked pairs per mask head: sum over columns of N - |masked rows of j|.
__global__ void __launch_bounds__(1024) count_kernel(int N, int causal,
                                                     const int32_t *__restrict__ lts,
                                                     const int32_t *__restrict__ lte,
                                                     const int32_t *__restrict__ uts,
                                                     const int32_t *__restrict__ ute,
                                                     unsigned long long *__restrict__ out) {
    __shared__ unsigned long long red[32];
    const int bm = blockIdx.x;
    const size_t row = static_cast<size_t>(bm) * N;
    unsigned long long acc = 0;
    for (int j = threadIdx.x; j < N; j += blockDim.x) {
        // Three intervals on [0, N): causal [0, j), LT, UT; measure of the union
        // by inclusion-exclusion.
        const int a0 = 0, b0 = causal ? j : 0;
        const int a1 = lts ? clampN(lts[row + j], N) : N, b1 = lte ? clampN(lte[row + j], N) : N;
        const int a2 = uts ? clampN(uts[row + j], N) : 0, b2 = ute ? clampN(ute[row + j], N) : 0;
        auto len = [](int a, int b) { return b > a ? b - a : 0; };
        auto len2 = [&](int a, int b, int c, int d) { return len(max(a, c), min(b, d)); };
        const int s1 = len(a0, b0) + len(a1, b1) + len(a2, b2);
        const int s2 = len2(a0, b0, a1, b1) + len2(a0, b0, a2, b2) + len2(a1, b1, a2, b2);
        const int s3 = len(max(a0, max(a1, a2)), min(b0, min(b1, b2)));
        acc += static_cast<unsigned long long>(N - (s1 - s2 + s3));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x < 32) {
        unsigned long long v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0ull;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (threadIdx.x == 0) out[bm] = v;
    }
}

}  // namespace

cudaError_t launch_classify(const Geometry &g, const MaskPtrs &m, const Workspace &ws,
                            cudaStream_t st) {
    // Chunks of 32 query tiles share each CTA's per-tile reduction; a small
    // map takes shorter chunks so that the grid still fills the GPU.
    int chunk = kClassifyChunk;
    const long long heads = static_cast<long long>(g.B) * g.Hm;
    while (chunk > 8 && heads * g.T * ((g.T + chunk - 1) / chunk) < 512) chunk /= 2;
    dim3 grid(g.T, (g.T + chunk - 1) / chunk, g.B * g.Hm);
    return launch_pdl(classify_kernel, grid, dim3(128), 0, st, g.N, g.T, g.Npad, g.Hm, g.causal,
                      chunk, m.lts, m.lte, m.uts, m.ute, ws.vec, ws.cls);
}

cudaError_t launch_fwd_lists(const Geometry &g, const Workspace &ws, cudaStream_t st) {
    const int rows = g.B * g.Hm * g.T;
    const int pair_rows = g.B * g.Hm * ((g.T + 1) / 2);
    const int list_blocks = (2 * rows + pair_rows + 31) / 32;
    const size_t smem = static_cast<size_t>((g.T + 1) / 2) * sizeof(int);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(fwd_lists_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(fwd_lists_kernel, dim3(list_blocks + g.B * g.Hm), dim3(1024), smem, st,
                      g.N, g.T, rows, pair_rows, list_blocks,
                      static_cast<const uint8_t *>(ws.cls), ws.fwd_list, ws.fwd_cnt, ws.bwd_list,
                      ws.bwd_cnt, ws.pair_list, ws.pair_cnt, ws.pair_order);
}

cudaError_t launch_validate_lists(const Geometry &g, const Workspace &ws, cudaStream_t st) {
    const long long rows = static_cast<long long>(g.B) * g.Hm * g.T;
    const long long pair_rows = static_cast<long long>(g.B) * g.Hm * ((g.T + 1) / 2);
    const long long jobs = 2 * rows + 2 * pair_rows;
    const unsigned blocks = static_cast<unsigned>((jobs * 32 + 255) / 256);
    return launch_pdl(validate_lists_kernel, dim3(blocks), dim3(256), 0, st, g.T,
                      static_cast<int>(rows), static_cast<int>(pair_rows), ws.fwd_list,
                      ws.fwd_cnt, ws.bwd_list, ws.bwd_cnt, ws.pair_list, ws.pair_cnt,
                      ws.pair_order);
}

cudaError_t launch_wait_selftest(uint64_t timeout_ns, cudaStream_t st) {
    wait_selftest_kernel<<<1, 32, 0, st>>>(timeout_ns);
    return cudaGetLastError();
}

cudaError_t launch_count(const Geometry &g, const MaskPtrs &m, unsigned long long *counts,
                         cudaStream_t st) {
    count_kernel<<<g.B * g.Hm, 1024, 0, st>>>(g.N, g.causal, m.lts, m.lte, m.uts, m.ute,
                                               counts);
    return cudaGetLastError();
}

unsigned read_clear_error_classify() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_err_classify, sizeof(v)) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_err_classify, &zero, sizeof(zero));
    return v;
}

}  // namespace fm
