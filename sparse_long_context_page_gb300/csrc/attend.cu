// Self-planning ragged paged attention over caller-given lists ("MOIRA:
// Mass-Oriented Indexing with Ragged Attention for Long-Context Decoding",
// abstract: the blocks plan their own work on the device from the list
// lengths, so no host plan runs and the step can be captured as one CUDA
// graph), with sequence-split partials merged by log-sum-exp (FlashDecoding,
// "Faster Flash Decoding" section 2).
//
// Work plan, computed by every block from device data only:
//   W = sum of the list lengths (block-wide scan of `lengths` in shared
//   memory); n = min(grid, W) active blocks; block b takes pages
//   [b*W/n, (b+1)*W/n) of the lists laid end to end and splits its range at
//   list boundaries into segments.  A segment's partial goes to slot b + u
//   (u = list index), which is unique.  The data path and the merges are
//   those of attend_core.cuh.
#include "attend_core.cuh"

namespace moira {

template <int kSlots, int kConsumerWarps>
__global__ void __launch_bounds__((kConsumerWarps + 1) * 32, kBlocksPerSm)
    k_attend(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
             const AttendArgs a)
{
    // Consumer warp w takes the pages whose range index is w modulo the warp
    // count, so with a slot count that is a multiple of it every slot belongs
    // to one warp, which waits on its rounds in order.  Otherwise a warp that
    // runs ahead could wait on a slot's parity one round early and match the
    // round before.
    static_assert(kSlots % kConsumerWarps == 0, "every ring slot belongs to one consumer warp");
    static_assert(kConsumerWarps >= kGroup, "the first 4 consumer warps own the (head, dims) slices");
    constexpr int kAttThreads = (kConsumerWarps + 1) * 32;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *stage = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    AttendSmem<kSlots, kConsumerWarps> &sm =
        *reinterpret_cast<AttendSmem<kSlots, kConsumerWarps> *>(stage + kSlots * kSlotBytes);
    int *s_off = reinterpret_cast<int *>(&sm + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int units = a.units;
    const WaitGuard wg{&sm.abort, a.status};

    attend_init(sm, &tmap_k, &tmap_v, a.status);
    pdl_trigger();
    pdl_wait();                               // lists and lengths come from k_select

    // ---- self-planning: exclusive scan of the list lengths -----------------
    {
        const int per = (units + kAttThreads - 1) / kAttThreads;
        const int ub = min(units, tid * per), ue = min(units, ub + per);
        int mine = 0;
        bool bad = false;
        // the first kLenCache lengths stay in registers for the second pass
        // (one global round trip fewer before the first page at small batch)
        auto length_of = [&](int u) {
            int len = a.lengths[u];
            if (len < 0 || len > a.max_pages) {
                bad = true;
                len = len < 0 ? 0 : a.max_pages;
            }
            return len;
        };
        int lv[kLenCache];
#pragma unroll
        for (int i = 0; i < kLenCache; ++i) {
            lv[i] = ub + i < ue ? length_of(ub + i) : 0;
            mine += lv[i];
        }
        for (int u = ub + kLenCache; u < ue; ++u) mine += length_of(u);
        if (bad) raise_status(a.status, kDevBadLen);
        int x = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        __shared__ int s_wsum[kConsumerWarps + 1];
        if (lane == 31) s_wsum[warp] = x;
        __syncthreads();
        int off = 0;
        for (int w = 0; w < warp; ++w) off += s_wsum[w];
        int run = off + x - mine;
#pragma unroll
        for (int i = 0; i < kLenCache; ++i) {
            if (ub + i < ue) s_off[ub + i] = run;
            run += lv[i];
        }
        for (int u = ub + kLenCache; u < ue; ++u) {
            s_off[u] = run;
            const int len = a.lengths[u];
            run += len < 0 ? 0 : (len > a.max_pages ? a.max_pages : len);
        }
        if (tid == kAttThreads - 1) s_off[units] = run;
    }
    __syncthreads();

    const long long W = s_off[units];
    const long long n = min(static_cast<long long>(gridDim.x), W);
    const int b = blockIdx.x;
    const long long g0 = b < n ? b * W / n : 0;
    const long long g1 = b < n ? (b + 1) * W / n : 0;

    if (warp == kConsumerWarps) {
        // entry k: its list (binary search in the offsets), the list entry and
        // the valid tokens (the partial tail page is the list's last entry)
        attend_produce(sm, stage, &tmap_k, &tmap_v, a, g0, g1, wg,
                       [&](long long k, int &u, int &ntok, int &pid) {
                           int lo = 0, hi = units;             // largest u with s_off[u] <= k
                           while (hi - lo > 1) {
                               const int mid = (lo + hi) >> 1;
                               if (s_off[mid] <= k) lo = mid; else hi = mid;
                           }
                           u = lo;
                           const int i = static_cast<int>(k - s_off[u]);
                           const int len = s_off[u + 1] - s_off[u];
                           pid = a.lists[static_cast<size_t>(u) * a.max_pages + i];
                           int L = a.seq_lens[u / a.hkv];
                           L = L < 0 ? 0 : (L > a.max_pages * kPageSize ? a.max_pages * kPageSize : L);
                           const int tail = L % kPageSize;
                           ntok = (i == len - 1 && tail) ? tail : kPageSize;
                       });
        return;
    }
    attend_consume(sm, stage, s_off, units, W, n, g0, g1, a, wg);
}

int attend_blocks_per_sm() { return kBlocksPerSm; }

// Per-device records of the shared-memory limit set for each block shape.
// They live at namespace scope with internal linkage: a static local of a
// function template would be one object shared by every library in the
// process that instantiates it (the load-balance build loaded next to this
// one), and the other library's kernels would then skip their own setting.
namespace {
std::atomic<int> g_attend_smem_seen[2][64];
}

template <int NS, int NW>
static cudaError_t launch_attend_shape(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                                       const AttendArgs &args, int blocks, cudaStream_t stream)
{
    const size_t smem = attend_smem_bytes<NS, NW>(args.units);
    cudaError_t e = raise_smem_limit(k_attend<NS, NW>, smem, g_attend_smem_seen[NW == kFewWarps ? 0 : 1]);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_attend<NS, NW>, dim3(blocks), dim3((NW + 1) * 32), smem, stream, tmap_k,
                      tmap_v, args);
}

cudaError_t launch_attend(const CUtensorMap &tmap_k, const CUtensorMap &tmap_v,
                          const AttendArgs &args, int blocks, cudaStream_t stream)
{
    if (args.units < kManyUnits)
        return launch_attend_shape<kFewSlots, kFewWarps>(tmap_k, tmap_v, args, blocks, stream);
    return launch_attend_shape<kManySlots, kManyWarps>(tmap_k, tmap_v, args, blocks, stream);
}

}  // namespace moira
