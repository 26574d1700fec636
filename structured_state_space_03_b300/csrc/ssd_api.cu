// ssd_api.cu -- the C ABI of libssd: argument checks, workspace, launch order.
//
// Launch sequence of one forward (all on the caller's stream, no host sync):
//   1. chunk states S_c and chunk decays      (per batch, head, chunk)
//   2. state passing h_{c+1} = a_c h_c + S_c  (sequential over chunks)
//   3. outputs: diagonal block + off-diagonal term + D skip
// following the block decomposition of "Mamba 模型" §4.1.
#include <stdio.h>
#include <stdarg.h>
#include <string.h>
#include <algorithm>
#include <mutex>
#include <vector>

#include "ssd_internal.cuh"

namespace ssd {

static thread_local char g_detail[512];
// Failure-detection test settings of this thread (ssd_test_set_fault).
static thread_local unsigned long long t_wait_ns;
static thread_local long long t_withhold = -1;

static ssd_status_t fail(ssd_status_t st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_detail, sizeof g_detail, fmt, ap);
    va_end(ap);
    return st;
}

static ssd_status_t ok()
{
    g_detail[0] = 0;
    return SSD_OK;
}

static __device__ unsigned int g_device_error;

// Device address of the error word on the current device (looked up once per device).
static unsigned int *device_error_word()
{
    static std::mutex mu;
    static unsigned int *addr[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<unsigned int *>(p);
    }
    return addr[dev];
}

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

static ssd_path_t choose_path(const Problem &pr);

// chunk states of the multi-kernel paths: [batch][nheads][nchunks], or
// [1][nheads][total_chunks] for packed sequences
static size_t state_units(const Problem &pr)
{
    return pr.chunks ? (size_t)pr.nheads * pr.total_chunks : (size_t)pr.batch * pr.nheads * pr.nchunks;
}

size_t workspace_bytes(const Problem &pr)
{
    if (choose_path(pr) == SSD_PATH_TCGEN05_FUSED) return fused_workspace_bytes(pr);
    const size_t units = state_units(pr);
    return align_up(units * pr.headdim * pr.dstate * sizeof(float), 256) +
           align_up(units * sizeof(float), 256) + 256;  // ..., the tile ticket
}

Workspace carve_workspace(const Problem &pr, void *base)
{
    const size_t units = state_units(pr);
    Workspace ws;
    ws.states = static_cast<float *>(base);
    ws.decay = reinterpret_cast<float *>(static_cast<char *>(base) +
                                         align_up(units * pr.headdim * pr.dstate * sizeof(float), 256));
    ws.ticket = reinterpret_cast<uint32_t *>(reinterpret_cast<char *>(ws.decay) + align_up(units * sizeof(float), 256));
    return ws;
}

// Evaluates a chunk longer than the fused kernels' 128-token tile as equal blocks of
// at most 128 tokens when a fused kernel then covers the sizes; false if none does.
static bool to_fused_blocks(Problem &pr)
{
    if (pr.chunk <= kFusedTile) return false;
    Problem q = pr;
    const int nb = (pr.chunk + kFusedTile - 1) / kFusedTile;
    q.chunk = (pr.chunk + nb - 1) / nb;
    q.nchunks = (pr.seqlen + q.chunk - 1) / q.chunk;
    if (!fused_supported(q)) return false;
    pr.chunk = q.chunk;
    pr.nchunks = q.nchunks;
    return true;
}

// Checks that need no pointer; fills the dimension fields of `pr`.
static ssd_status_t check_dims(Problem &pr, int batch, int seqlen, int nheads, int headdim, int ngroups,
                               int dstate, int chunk, ssd_dtype_t dtype)
{
    if (batch <= 0 || seqlen <= 0 || nheads <= 0 || headdim <= 0 || ngroups <= 0 || dstate <= 0 || chunk <= 0)
        return fail(SSD_ERR_INVALID_ARG,
                    "every dimension must be positive (batch=%d seqlen=%d nheads=%d headdim=%d ngroups=%d "
                    "dstate=%d chunk=%d)", batch, seqlen, nheads, headdim, ngroups, dstate, chunk);
    if (nheads % ngroups != 0)
        return fail(SSD_ERR_INVALID_ARG, "nheads (%d) must be a multiple of ngroups (%d)", nheads, ngroups);
    if (dtype != SSD_DTYPE_F32 && dtype != SSD_DTYPE_BF16)
        return fail(SSD_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (chunk > kMaxChunk)
        return fail(SSD_ERR_UNSUPPORTED, "chunk %d exceeds %d", chunk, kMaxChunk);
    if (headdim > kMaxHeaddim || dstate > kMaxDstate)
        return fail(SSD_ERR_UNSUPPORTED, "headdim %d / dstate %d exceed %d / %d", headdim, dstate, kMaxHeaddim,
                    kMaxDstate);
    if (nheads > 65535 || batch > 65535)
        return fail(SSD_ERR_UNSUPPORTED, "nheads and batch must each be <= 65535");
    pr.batch = batch;
    pr.seqlen = seqlen;
    pr.nheads = nheads;
    pr.headdim = headdim;
    pr.ngroups = ngroups;
    pr.dstate = dstate;
    pr.chunk = chunk;
    pr.nchunks = (seqlen + chunk - 1) / chunk;
    pr.dtype = dtype;
    // The block decomposition is exact for any chunk length, so a chunk longer than the
    // fused kernels' 128-token tile is evaluated as equal blocks of at most 128 tokens
    // where a fused kernel covers the sizes and is the faster choice: at dstate 64 (the
    // pipelined fused kernels), and wherever the three-kernel tcgen05 path cannot take the
    // requested length.  At dstate 128 the three-kernel path at the requested length
    // measured faster than the one-unit-at-a-time fused kernel at 128-token blocks (0.27
    // against 0.32 ms on 1 x 8192 tokens, 80 heads x 64, chunk 256).  The results differ
    // from the requested length only in rounding.
    if (dstate == 64 || !tc_supported(pr)) to_fused_blocks(pr);
    return SSD_OK;
}

static bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

static ssd_status_t check_pointers(const Problem &pr)
{
    if (!pr.x || !pr.dt || !pr.A || !pr.B || !pr.C || !pr.y)
        return fail(SSD_ERR_INVALID_ARG, "x, dt, A, B, C and y must be non-NULL");
    const size_t el = pr.dtype == SSD_DTYPE_BF16 ? 16 : 4;
    if (!aligned(pr.x, el) || !aligned(pr.B, el) || !aligned(pr.C, el) || !aligned(pr.y, el))
        return fail(SSD_ERR_INVALID_ARG, "x, B, C and y must be %zu-byte aligned", el);
    if (!aligned(pr.dt, 4) || !aligned(pr.A, 4) || (pr.D && !aligned(pr.D, 4)) ||
        (pr.init_state && !aligned(pr.init_state, 4)) || (pr.final_state && !aligned(pr.final_state, 4)))
        return fail(SSD_ERR_INVALID_ARG, "fp32 tensors must be 4-byte aligned");
    return SSD_OK;
}

static ssd_path_t choose_path(const Problem &pr)
{
    if (fused_supported(pr)) return SSD_PATH_TCGEN05_FUSED;
    return tc_supported(pr) ? SSD_PATH_TCGEN05 : SSD_PATH_SIMT;
}

static const char *kernel_names(const Problem &pr)
{
    switch (choose_path(pr)) {
    case SSD_PATH_SIMT: return "chunk_state_simt,state_pass,chunk_out_simt";
    case SSD_PATH_TCGEN05: return "chunk_state_tc,state_pass_hilo,chunk_out_tc";
    case SSD_PATH_TCGEN05_FUSED:
        return seq_supported(pr) ? "ssd_seq_pipe_tc" : (pr.dstate == 64 ? "ssd_fused_pipe_tc" : "ssd_fused_tc");
    default: return "";
    }
}

static ssd_status_t run(const Problem &pr_in, void *workspace, cudaStream_t s)
{
    Problem pr = pr_in;
    pr.wait_ns = t_wait_ns ? t_wait_ns : 2000000000ull;
    pr.withhold = t_withhold;
    pr.err_word = device_error_word();
    if (!pr.err_word) return fail(SSD_ERR_CUDA, "cannot resolve the device error word");
    const ssd_path_t path = choose_path(pr);
    profile_forward_begin();
    if (path == SSD_PATH_TCGEN05_FUSED) {
        cudaError_t e = launch_fused_tc(pr, workspace, s);
        if (e != cudaSuccess) return fail(SSD_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
        return ok();
    }
    const Workspace ws = carve_workspace(pr, workspace);
    const bool tc = path == SSD_PATH_TCGEN05;
    cudaError_t e = tc ? launch_chunk_state_tc(pr, ws, s) : launch_chunk_state_simt(pr, ws, s);
    if (e == cudaSuccess) e = launch_state_pass(pr, ws, s, tc);
    if (e == cudaSuccess) e = tc ? launch_chunk_out_tc(pr, ws, s) : launch_chunk_out_simt(pr, ws, s);
    if (e != cudaSuccess) return fail(SSD_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    return ok();
}

static ssd_status_t make_problem(Problem &pr, const void *x, const float *dt, const float *A, const void *B,
                                 const void *C, const float *D, const float *init_state, void *y,
                                 float *final_state, int batch, int seqlen, int nheads, int headdim, int ngroups,
                                 int dstate, int chunk, ssd_dtype_t dtype)
{
    memset(&pr, 0, sizeof pr);
    ssd_status_t st = check_dims(pr, batch, seqlen, nheads, headdim, ngroups, dstate, chunk, dtype);
    if (st != SSD_OK) return st;
    pr.x = x;
    pr.dt = dt;
    pr.A = A;
    pr.B = B;
    pr.C = C;
    pr.D = D;
    pr.init_state = init_state;
    pr.y = y;
    pr.final_state = final_state;
    return check_pointers(pr);
}

}  // namespace ssd

using namespace ssd;

extern "C" {

ssd_status_t ssd_fwd_workspace_size(int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate,
                                    int chunk, ssd_dtype_t dtype, size_t *bytes)
{
    if (!bytes) return fail(SSD_ERR_INVALID_ARG, "bytes must be non-NULL");
    Problem pr;
    memset(&pr, 0, sizeof pr);
    ssd_status_t st = check_dims(pr, batch, seqlen, nheads, headdim, ngroups, dstate, chunk, dtype);
    if (st != SSD_OK) return st;
    *bytes = workspace_bytes(pr);
    return ok();
}

ssd_path_t ssd_fwd_path(int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate, int chunk,
                        ssd_dtype_t dtype)
{
    Problem pr;
    memset(&pr, 0, sizeof pr);
    if (check_dims(pr, batch, seqlen, nheads, headdim, ngroups, dstate, chunk, dtype) != SSD_OK)
        return SSD_PATH_NONE;
    return choose_path(pr);
}

int ssd_fwd_block(int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate, int chunk,
                  ssd_dtype_t dtype)
{
    Problem pr;
    memset(&pr, 0, sizeof pr);
    if (check_dims(pr, batch, seqlen, nheads, headdim, ngroups, dstate, chunk, dtype) != SSD_OK) return -1;
    return pr.chunk;
}

int ssd_fwd_kernels(int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate, int chunk,
                    ssd_dtype_t dtype, char *names, size_t names_len)
{
    Problem pr;
    memset(&pr, 0, sizeof pr);
    if (check_dims(pr, batch, seqlen, nheads, headdim, ngroups, dstate, chunk, dtype) != SSD_OK) return -1;
    const char *list = kernel_names(pr);
    if (names && names_len) snprintf(names, names_len, "%s", list);
    int count = list[0] ? 1 : 0;
    for (const char *c = list; *c; ++c) count += *c == ',';
    return count;
}

ssd_status_t ssd_profile_events(void *const *events, int count)
{
    if (!events || count <= 0) {
        profile_set(nullptr, 0);
        return ok();
    }
    if (count > kMaxProfileEvents) return fail(SSD_ERR_INVALID_ARG, "at most %d profiling events", kMaxProfileEvents);
    for (int i = 0; i < count; ++i)
        if (!events[i]) return fail(SSD_ERR_INVALID_ARG, "profiling event %d is NULL", i);
    profile_set(events, count);
    return ok();
}

ssd_status_t ssd_fwd_ws(const void *x, const float *dt, const float *A, const void *B, const void *C,
                        const float *D, const float *init_state, void *y, float *final_state, int batch,
                        int seqlen, int nheads, int headdim, int ngroups, int dstate, int chunk,
                        ssd_dtype_t dtype, void *workspace, size_t workspace_bytes_given, void *stream)
{
    Problem pr;
    ssd_status_t st = make_problem(pr, x, dt, A, B, C, D, init_state, y, final_state, batch, seqlen, nheads,
                                   headdim, ngroups, dstate, chunk, dtype);
    if (st != SSD_OK) return st;
    const size_t need = workspace_bytes(pr);
    if (!workspace || !aligned(workspace, 256))
        return fail(SSD_ERR_INVALID_ARG, "workspace must be non-NULL and 256-byte aligned");
    if (workspace_bytes_given < need)
        return fail(SSD_ERR_INVALID_ARG, "workspace too small: %zu bytes given, %zu needed", workspace_bytes_given,
                    need);
    return run(pr, workspace, static_cast<cudaStream_t>(stream));
}

ssd_status_t ssd_fwd(const void *x, const float *dt, const float *A, const void *B, const void *C, const float *D,
                     const float *init_state, void *y, float *final_state, int batch, int seqlen, int nheads,
                     int headdim, int ngroups, int dstate, int chunk, ssd_dtype_t dtype, void *stream)
{
    Problem pr;
    ssd_status_t st = make_problem(pr, x, dt, A, B, C, D, init_state, y, final_state, batch, seqlen, nheads,
                                   headdim, ngroups, dstate, chunk, dtype);
    if (st != SSD_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t need = workspace_bytes(pr);
    void *ws = nullptr;
    cudaError_t e = cudaMallocAsync(&ws, need, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(e == cudaErrorMemoryAllocation ? SSD_ERR_NO_MEMORY : SSD_ERR_CUDA,
                    "workspace allocation of %zu bytes failed: %s", need, cudaGetErrorString(e));
    }
    st = run(pr, ws, s);
    e = cudaFreeAsync(ws, s);
    if (st == SSD_OK && e != cudaSuccess)
        return fail(SSD_ERR_CUDA, "workspace release failed: %s", cudaGetErrorString(e));
    return st;
}

ssd_status_t ssd_fwd_varlen(const void *x, const float *dt, const float *A, const void *B, const void *C,
                            const float *D, const int *cu_seqlens, int nseq, const float *init_state, void *y,
                            float *final_state, int nheads, int headdim, int ngroups, int dstate, int chunk,
                            ssd_dtype_t dtype, void *stream)
{
    if (!cu_seqlens || nseq <= 0) return fail(SSD_ERR_INVALID_ARG, "cu_seqlens must be non-NULL and nseq positive");
    if (cu_seqlens[0] != 0) return fail(SSD_ERR_INVALID_ARG, "cu_seqlens[0] must be 0 (got %d)", cu_seqlens[0]);
    for (int q = 0; q < nseq; ++q)
        if (cu_seqlens[q + 1] < cu_seqlens[q])
            return fail(SSD_ERR_INVALID_ARG, "cu_seqlens decreases at %d (%d -> %d)", q, cu_seqlens[q],
                        cu_seqlens[q + 1]);
    const int total = cu_seqlens[nseq];
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t state_el = (size_t)nheads * headdim * dstate;
    if (total == 0) {  // only empty sequences: the final states are the initial states
        Problem chk;
        memset(&chk, 0, sizeof chk);
        ssd_status_t st = check_dims(chk, nseq, 1, nheads, headdim, ngroups, dstate, chunk, dtype);
        if (st != SSD_OK) return st;
        cudaError_t e = cudaSuccess;
        if (final_state && final_state != init_state)
            e = init_state ? cudaMemcpyAsync(final_state, init_state, nseq * state_el * sizeof(float),
                                             cudaMemcpyDeviceToDevice, s)
                           : cudaMemsetAsync(final_state, 0, nseq * state_el * sizeof(float), s);
        return e == cudaSuccess ? ok() : fail(SSD_ERR_CUDA, "final state copy failed: %s", cudaGetErrorString(e));
    }
    Problem pr;
    ssd_status_t st = make_problem(pr, x, dt, A, B, C, D, init_state, y, final_state, nseq, total, nheads, headdim,
                                   ngroups, dstate, chunk, dtype);
    if (st != SSD_OK) return st;
    // chunk table in chunk-major order (a counting sort over the chunk index), in chunks of
    // the evaluated block length
    chunk = pr.chunk;
    std::vector<int> nchunk(nseq);
    int max_nc = 0;
    size_t total_chunks = 0;
    for (int q = 0; q < nseq; ++q) {
        const int len = cu_seqlens[q + 1] - cu_seqlens[q];
        nchunk[q] = (len + chunk - 1) / chunk;
        max_nc = std::max(max_nc, nchunk[q]);
        total_chunks += nchunk[q];
    }
    std::vector<size_t> cursor(max_nc + 1, 0);
    for (int q = 0; q < nseq; ++q)
        for (int c = 0; c < nchunk[q]; ++c) ++cursor[c + 1];
    for (int c = 0; c < max_nc; ++c) cursor[c + 1] += cursor[c];
    std::vector<ChunkDesc> table(total_chunks);
    size_t gbase = 0;
    for (int q = 0; q < nseq; ++q) {
        const int len = cu_seqlens[q + 1] - cu_seqlens[q];
        for (int c = 0; c < nchunk[q]; ++c) {
            ChunkDesc &d = table[cursor[c]++];
            d.b = q;
            d.c = c;
            d.gchunk = (int)(gbase + c);
            d.tok0 = cu_seqlens[q] + c * chunk;
            d.len = std::min(chunk, len - c * chunk);
            d.last = c == nchunk[q] - 1;
            d.pad0 = d.pad1 = 0;
        }
        gbase += nchunk[q];
    }
    if (total_chunks > (size_t)INT32_MAX) return fail(SSD_ERR_UNSUPPORTED, "too many chunks for the packed layout");
    pr.total_chunks = (int)total_chunks;
    pr.chunks = reinterpret_cast<const ChunkDesc *>(1);  // marks the packed layout for the size query below
    // the multi-kernel paths also need each sequence's first chunk (sequence-major numbering)
    const bool fused = choose_path(pr) == SSD_PATH_TCGEN05_FUSED;
    std::vector<int> seq_first(fused ? 0 : nseq + 1);
    if (!fused) {
        seq_first[0] = 0;
        for (int q = 0; q < nseq; ++q) seq_first[q + 1] = seq_first[q] + nchunk[q];
    }
    const size_t main_bytes = align_up(workspace_bytes(pr), 256);
    const size_t table_bytes = align_up(total_chunks * sizeof(ChunkDesc), 256);
    const size_t need = main_bytes + table_bytes + seq_first.size() * sizeof(int);
    void *ws = nullptr;
    cudaError_t e = cudaMallocAsync(&ws, need, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(e == cudaErrorMemoryAllocation ? SSD_ERR_NO_MEMORY : SSD_ERR_CUDA,
                    "workspace allocation of %zu bytes failed: %s", need, cudaGetErrorString(e));
    }
    ChunkDesc *dtab = reinterpret_cast<ChunkDesc *>(static_cast<char *>(ws) + main_bytes);
    int *dfirst = reinterpret_cast<int *>(static_cast<char *>(ws) + main_bytes + table_bytes);
    e = cudaMemcpyAsync(dtab, table.data(), total_chunks * sizeof(ChunkDesc), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess && !fused)
        e = cudaMemcpyAsync(dfirst, seq_first.data(), seq_first.size() * sizeof(int), cudaMemcpyHostToDevice, s);
    // empty sequences get no unit: their final state is their initial state
    for (int q = 0; q < nseq && e == cudaSuccess; ++q) {
        if (nchunk[q] != 0 || !final_state || final_state == init_state) continue;
        e = init_state ? cudaMemcpyAsync(final_state + q * state_el, init_state + q * state_el,
                                         state_el * sizeof(float), cudaMemcpyDeviceToDevice, s)
                       : cudaMemsetAsync(final_state + q * state_el, 0, state_el * sizeof(float), s);
    }
    if (e == cudaSuccess) {
        pr.chunks = dtab;
        pr.seq_first = fused ? nullptr : dfirst;
        st = run(pr, ws, s);
    } else {
        st = fail(SSD_ERR_CUDA, "chunk table upload failed: %s", cudaGetErrorString(e));
    }
    e = cudaFreeAsync(ws, s);
    if (st == SSD_OK && e != cudaSuccess)
        return fail(SSD_ERR_CUDA, "workspace release failed: %s", cudaGetErrorString(e));
    return st;
}

ssd_status_t ssd_fwd_pre(const void *x, const float *dt, const float *dt_bias, int pre_flags, const float *A,
                         const void *B, const void *C, const float *D, const float *init_state, void *y,
                         float *final_state, int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate,
                         int chunk, ssd_dtype_t dtype, void *stream)
{
    if (pre_flags & ~(SSD_PRE_SOFTPLUS | SSD_PRE_ZOH)) return fail(SSD_ERR_INVALID_ARG, "unknown pre_flags 0x%x", pre_flags);
    if (dt_bias && !aligned(dt_bias, 4)) return fail(SSD_ERR_INVALID_ARG, "dt_bias must be 4-byte aligned");
    Problem pr;
    ssd_status_t st = make_problem(pr, x, dt, A, B, C, D, init_state, y, final_state, batch, seqlen, nheads,
                                   headdim, ngroups, dstate, chunk, dtype);
    if (st != SSD_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t main_bytes = (workspace_bytes(pr) + 255) / 256 * 256;
    const size_t n = (size_t)batch * seqlen * nheads;
    const size_t col = (n * sizeof(float) + 255) / 256 * 256;
    const bool zoh = (pre_flags & SSD_PRE_ZOH) != 0;
    const size_t need = main_bytes + col * (zoh ? 2 : 1);
    void *ws = nullptr;
    cudaError_t e = cudaMallocAsync(&ws, need, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(e == cudaErrorMemoryAllocation ? SSD_ERR_NO_MEMORY : SSD_ERR_CUDA,
                    "workspace allocation of %zu bytes failed: %s", need, cudaGetErrorString(e));
    }
    float *dt_eff = reinterpret_cast<float *>(static_cast<char *>(ws) + main_bytes);
    float *scale = zoh ? reinterpret_cast<float *>(static_cast<char *>(ws) + main_bytes + col) : nullptr;
    e = launch_pre(dt, dt_bias, A, pre_flags, dt_eff, scale, batch, seqlen, nheads, s);
    if (e != cudaSuccess) {
        cudaFreeAsync(ws, s);
        return fail(SSD_ERR_CUDA, "pre-step launch failed: %s", cudaGetErrorString(e));
    }
    pr.dt = dt_eff;
    pr.dtin = scale;
    st = run(pr, ws, s);
    e = cudaFreeAsync(ws, s);
    if (st == SSD_OK && e != cudaSuccess)
        return fail(SSD_ERR_CUDA, "workspace release failed: %s", cudaGetErrorString(e));
    return st;
}

// ---------------------------------------------------------------------------
// Forward without any allocation, for callers that may not allocate device
// memory: processes whose device memory is handed in full to a framework-owned
// pool, plugins hosted by such runtimes, and latency-critical loops that cannot
// afford an allocator call (it can synchronise the device or fail under memory
// pressure).  Its scratch is the fixed array below, which every device that
// loads this library keeps until the process exits.
// ---------------------------------------------------------------------------

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device.  The first call
// on a device looks it up (cudaGetSymbolAddress); later calls reuse it.
static ssd_status_t noalloc_scratch(void **out)
{
    static std::mutex mu;
    static void *addr[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SSD_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(SSD_ERR_UNSUPPORTED, "device ordinal %d beyond 63", dev);
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return fail(SSD_ERR_CUDA, "cudaGetSymbolAddress of the fixed scratch failed: %s", cudaGetErrorString(e));
        addr[dev] = p;
    }
    *out = addr[dev];
    return SSD_OK;
}

ssd_status_t ssd_fwd_noalloc(const void *x, const float *dt, const float *A, const void *B, const void *C,
                             const float *D, const float *init_state, void *y, float *final_state, int batch,
                             int seqlen, int nheads, int headdim, int ngroups, int dstate, int chunk,
                             ssd_dtype_t dtype, void *stream)
{
    Problem pr;
    ssd_status_t st = make_problem(pr, x, dt, A, B, C, D, init_state, y, final_state, batch, seqlen, nheads,
                                   headdim, ngroups, dstate, chunk, dtype);
    if (st != SSD_OK) return st;
    // only the fused kernels run here: a longer chunk at dstate 128 as 128-token blocks too
    if (choose_path(pr) != SSD_PATH_TCGEN05_FUSED) to_fused_blocks(pr);
    if (choose_path(pr) != SSD_PATH_TCGEN05_FUSED)
        return fail(SSD_ERR_UNSUPPORTED,
                    "ssd_fwd_noalloc runs the fused bf16 kernel only (bf16, headdim 64 or 128, dstate 64 or "
                    "128)");
    const size_t need = workspace_bytes(pr);
    if (need > kNoAllocScratchBytes)
        return fail(SSD_ERR_UNSUPPORTED,
                    "problem needs %zu bytes of scratch; the fixed scratch of ssd_fwd_noalloc holds %zu bytes",
                    need, kNoAllocScratchBytes);
    void *scratch = nullptr;
    if ((st = noalloc_scratch(&scratch)) != SSD_OK) return st;
    return run(pr, scratch, static_cast<cudaStream_t>(stream));
}

// Host-buffer entry: the problem is cut into at most kHostParts parts.
constexpr int kHostParts = 8;

// Copy streams, events and device memory pool of the host-buffer entry, one set
// per device, made on first use; calls on one device take its lock for their
// whole duration.  The pool keeps the memory of earlier calls (its release
// threshold is unlimited), so a call in a loop does not map its ~2x input size
// of device memory again each time; the process's default pool is left as it is.
struct HostCopyRes {
    std::mutex mu;
    bool made = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t ev[2 * kHostParts + 2];
    cudaMemPool_t pool = nullptr;
};

static ssd_status_t host_copy_res(HostCopyRes **res)
{
    static std::mutex mu;
    static HostCopyRes all[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SSD_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= 64) return fail(SSD_ERR_UNSUPPORTED, "device ordinal %d beyond 64", dev);
    std::lock_guard<std::mutex> lock(mu);
    HostCopyRes &r = all[dev];
    if (!r.made) {
        if ((e = cudaStreamCreateWithFlags(&r.in, cudaStreamNonBlocking)) == cudaSuccess)
            e = cudaStreamCreateWithFlags(&r.out, cudaStreamNonBlocking);
        for (int k = 0; k < 2 * kHostParts + 2 && e == cudaSuccess; ++k)
            e = cudaEventCreateWithFlags(&r.ev[k], cudaEventDisableTiming);
        if (e == cudaSuccess) {
            cudaMemPoolProps props;
            memset(&props, 0, sizeof props);
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            e = cudaMemPoolCreate(&r.pool, &props);
            uint64_t keep = ~uint64_t(0);
            if (e == cudaSuccess) e = cudaMemPoolSetAttribute(r.pool, cudaMemPoolAttrReleaseThreshold, &keep);
        }
        if (e != cudaSuccess)
            return fail(SSD_ERR_CUDA, "copy stream, event or memory pool creation failed: %s", cudaGetErrorString(e));
        r.made = true;
    }
    *res = &r;
    return SSD_OK;
}

ssd_status_t ssd_fwd_host(const void *x, const float *dt, const float *A, const void *B, const void *C,
                          const float *D, const float *init_state, void *y, float *final_state, int batch,
                          int seqlen, int nheads, int headdim, int ngroups, int dstate, int chunk,
                          ssd_dtype_t dtype, void *stream)
{
    Problem pr;
    memset(&pr, 0, sizeof pr);
    ssd_status_t st = check_dims(pr, batch, seqlen, nheads, headdim, ngroups, dstate, chunk, dtype);
    if (st != SSD_OK) return st;
    chunk = pr.chunk;  // the evaluated block length: the parts are cut at its multiples
    if (!x || !dt || !A || !B || !C || !y)
        return fail(SSD_ERR_INVALID_ARG, "x, dt, A, B, C and y must be non-NULL");
    HostCopyRes *res = nullptr;
    if ((st = host_copy_res(&res)) != SSD_OK) return st;
    std::lock_guard<std::mutex> lock(res->mu);
    cudaStream_t s = static_cast<cudaStream_t>(stream), sin = res->in, sout = res->out;
    const size_t el = dtype == SSD_DTYPE_BF16 ? 2 : 4;
    const size_t H = nheads, P = headdim, G = ngroups, N = dstate;
    const size_t tok = (size_t)batch * seqlen;
    const size_t n_x = tok * H * P, n_dt = tok * H, n_bc = tok * G * N;
    const size_t n_state = (size_t)batch * H * P * N;

    // The problem is cut into parts whose copies and compute overlap: uploads on
    // one stream, the scan on `stream`, downloads on another (the two copy
    // directions run at once).  kHostParts or more batch elements: groups of
    // them.  Fewer: each batch element in whole-chunk token ranges, the state of
    // one range carried into the next in place (init_state == final_state).
    struct Part { int b0, nb, t0, nt; };
    Part parts[kHostParts];
    int np = 0;
    const int nc = pr.nchunks;
    // parts start at token boundaries: keep their device addresses 16-byte aligned
    const bool splittable = (H * P * el) % 16 == 0 && (G * N * el) % 16 == 0;
    if (!splittable) {
        parts[np++] = {0, batch, 0, seqlen};
    } else if (batch >= kHostParts) {
        for (int k = 0; k < kHostParts; ++k) {
            const int b0 = (int)((long long)batch * k / kHostParts), b1 = (int)((long long)batch * (k + 1) / kHostParts);
            parts[np++] = {b0, b1 - b0, 0, seqlen};
        }
    } else {
        const int per = std::max(1, std::min(nc, kHostParts / batch));  // token ranges per batch element
        // The problem's first upload and last download overlap nothing, so its first and
        // last ranges are short (1/16 of a batch element's chunks); the others share the rest.
        const int small = std::max(1, nc / 16);
        for (int b = 0; b < batch; ++b) {
            const bool lo_small = b == 0 && per >= 2, hi_small = b == batch - 1 && per >= (lo_small ? 3 : 2);
            const int nsmall = (lo_small ? 1 : 0) + (hi_small ? 1 : 0);
            const int c_lo = lo_small ? small : 0, c_hi = hi_small ? nc - small : nc;
            const bool shaped = nsmall > 0 && c_hi - c_lo >= per - nsmall;
            int cut[kHostParts + 1];
            cut[0] = 0;
            cut[per] = nc;
            if (shaped) {
                const int k0 = lo_small ? 1 : 0, m = per - nsmall;  // m equal ranges over [c_lo, c_hi)
                if (lo_small) cut[1] = c_lo;
                for (int k = 0; k < m; ++k) cut[k0 + k + 1] = c_lo + (c_hi - c_lo) * (k + 1) / m;
            } else {
                for (int k = 1; k < per; ++k) cut[k] = nc * k / per;
            }
            for (int k = 0; k < per; ++k)
                parts[np++] = {b, 1, cut[k] * chunk, std::min(seqlen, cut[k + 1] * chunk) - cut[k] * chunk};
        }
    }
    const bool chained = np > 1 && parts[0].nb == 1 && np > batch;  // token ranges carry the state
    size_t ws_need = 0;
    for (int k = 0; k < np; ++k) {
        Problem q = pr;
        q.batch = parts[k].nb;
        q.seqlen = parts[k].nt;
        q.nchunks = (parts[k].nt + chunk - 1) / chunk;
        ws_need = std::max(ws_need, workspace_bytes(q));
    }
    // one device block: x | B | C | y | dt | A | D | state in | state out | workspace
    const bool need_state = final_state || chained;
    size_t off[11];
    size_t sizes[10] = {n_x * el, n_bc * el, n_bc * el, n_x * el, n_dt * 4, H * 4, D ? H * 4 : 0,
                        init_state ? n_state * 4 : 0, need_state ? n_state * 4 : 0, ws_need};
    off[0] = 0;
    for (int i = 0; i < 10; ++i) off[i + 1] = align_up(off[i] + sizes[i], 256);
    char *dev = nullptr;
    cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void **>(&dev), off[10], res->pool, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(e == cudaErrorMemoryAllocation ? SSD_ERR_NO_MEMORY : SSD_ERR_CUDA,
                    "device allocation of %zu bytes failed: %s", off[10], cudaGetErrorString(e));
    }
    cudaEvent_t *ev = res->ev;
    cudaEvent_t ev_alloc = ev[2 * np], ev_out = ev[2 * np + 1];
    char *const hx = (char *)x, *const hy = (char *)y, *const hB = (char *)B, *const hC = (char *)C;
    const char *hdt = reinterpret_cast<const char *>(dt);
    auto up = [&](size_t doff, const void *src, size_t bytes) {
        if (e == cudaSuccess && bytes) e = cudaMemcpyAsync(dev + doff, src, bytes, cudaMemcpyHostToDevice, sin);
    };
    // the allocation is ordered on `stream`; the copy streams wait for it
    if (e == cudaSuccess) e = cudaEventRecord(ev_alloc, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(sin, ev_alloc, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(sout, ev_alloc, 0);
    up(off[5], A, sizes[5]);
    up(off[6], D, sizes[6]);
    up(off[7], init_state, sizes[7]);
    for (int k = 0; k < np && e == cudaSuccess && st == SSD_OK; ++k) {
        const Part &pt = parts[k];
        const size_t t_first = (size_t)pt.b0 * seqlen + pt.t0;       // first token of the part
        const size_t t_count = (size_t)pt.nb * pt.nt;
        const size_t ox = t_first * H * P * el, obc = t_first * G * N * el, odt = t_first * H * 4;
        up(off[0] + ox, hx + ox, t_count * H * P * el);
        up(off[1] + obc, hB + obc, t_count * G * N * el);
        up(off[2] + obc, hC + obc, t_count * G * N * el);
        up(off[4] + odt, hdt + odt, t_count * H * 4);
        if (e == cudaSuccess) e = cudaEventRecord(ev[2 * k], sin);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev[2 * k], 0);
        if (e != cudaSuccess) break;
        Problem q = pr;
        q.batch = pt.nb;
        q.seqlen = pt.nt;
        q.nchunks = (pt.nt + chunk - 1) / chunk;
        q.x = dev + off[0] + ox;
        q.B = dev + off[1] + obc;
        q.C = dev + off[2] + obc;
        q.y = dev + off[3] + ox;
        q.dt = reinterpret_cast<const float *>(dev + off[4] + odt);
        q.A = reinterpret_cast<const float *>(dev + off[5]);
        q.D = D ? reinterpret_cast<const float *>(dev + off[6]) : nullptr;
        const size_t ost = (size_t)pt.b0 * H * P * N * 4;
        float *state_out = need_state ? reinterpret_cast<float *>(dev + off[8] + ost) : nullptr;
        if (chained && pt.t0 > 0)
            q.init_state = state_out;  // carried in place from the previous token range
        else
            q.init_state = init_state ? reinterpret_cast<const float *>(dev + off[7] + ost) : nullptr;
        q.final_state = state_out;
        st = run(q, dev + off[9], s);
        if (st != SSD_OK) break;
        if ((e = cudaEventRecord(ev[2 * k + 1], s)) == cudaSuccess) e = cudaStreamWaitEvent(sout, ev[2 * k + 1], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(hy + ox, dev + off[3] + ox, t_count * H * P * el, cudaMemcpyDeviceToHost, sout);
    }
    if (e == cudaSuccess && st == SSD_OK && final_state)
        e = cudaMemcpyAsync(final_state, dev + off[8], sizes[8], cudaMemcpyDeviceToHost, sout);
    // the block is released on `stream` after both copy streams are done with it
    cudaError_t e2 = cudaEventRecord(ev_out, sout);
    if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(s, ev_out, 0);
    cudaError_t e3 = cudaEventRecord(ev_alloc, sin);
    if (e3 == cudaSuccess) e3 = cudaStreamWaitEvent(s, ev_alloc, 0);
    cudaError_t ef = cudaFreeAsync(dev, s);
    cudaError_t es = cudaStreamSynchronize(s);
    if (st != SSD_OK) return st;
    if (e == cudaSuccess) e = e2 != cudaSuccess ? e2 : e3;
    if (e != cudaSuccess || ef != cudaSuccess || es != cudaSuccess)
        return fail(SSD_ERR_CUDA, "host-buffer forward failed: %s",
                    cudaGetErrorString(e != cudaSuccess ? e : (ef != cudaSuccess ? ef : es)));
    return ssd_check_device_status(stream);
}

ssd_status_t ssd_step(const void *x, const float *dt, const float *A, const void *B, const void *C, const float *D,
                      float *state, void *y, int batch, int nheads, int headdim, int ngroups, int dstate,
                      ssd_dtype_t dtype, void *stream)
{
    if (batch <= 0 || nheads <= 0 || headdim <= 0 || ngroups <= 0 || dstate <= 0)
        return fail(SSD_ERR_INVALID_ARG, "every dimension must be positive (batch=%d nheads=%d headdim=%d ngroups=%d "
                    "dstate=%d)", batch, nheads, headdim, ngroups, dstate);
    if (nheads % ngroups != 0)
        return fail(SSD_ERR_INVALID_ARG, "nheads (%d) must be a multiple of ngroups (%d)", nheads, ngroups);
    if (dtype != SSD_DTYPE_F32 && dtype != SSD_DTYPE_BF16) return fail(SSD_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (!x || !dt || !A || !B || !C || !state || !y)
        return fail(SSD_ERR_INVALID_ARG, "x, dt, A, B, C, state and y must be non-NULL");
    const size_t el = dtype == SSD_DTYPE_BF16 ? 2 : 4;
    if (!aligned(x, el) || !aligned(B, el) || !aligned(C, el) || !aligned(y, el) || !aligned(dt, 4) ||
        !aligned(A, 4) || (D && !aligned(D, 4)) || !aligned(state, 4))
        return fail(SSD_ERR_INVALID_ARG, "pointers must be aligned to their element size");
    const cudaError_t e = launch_step(x, dt, A, B, C, D, state, y, batch, nheads, headdim, ngroups, dstate, dtype,
                                      static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(SSD_ERR_CUDA, "ssd_step launch failed: %s", cudaGetErrorString(e));
    return ok();
}

static ssd_status_t make_bwd_problem(BwdProblem &p, int batch, int seqlen, int nheads, int headdim, int ngroups,
                                     int dstate, ssd_dtype_t dtype)
{
    memset(&p, 0, sizeof p);
    if (batch <= 0 || seqlen <= 0 || nheads <= 0 || headdim <= 0 || ngroups <= 0 || dstate <= 0)
        return fail(SSD_ERR_INVALID_ARG,
                    "every dimension must be positive (batch=%d seqlen=%d nheads=%d headdim=%d ngroups=%d dstate=%d)",
                    batch, seqlen, nheads, headdim, ngroups, dstate);
    if (nheads % ngroups != 0)
        return fail(SSD_ERR_INVALID_ARG, "nheads (%d) must be a multiple of ngroups (%d)", nheads, ngroups);
    if (dtype != SSD_DTYPE_F32 && dtype != SSD_DTYPE_BF16) return fail(SSD_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (headdim > kBwdMaxHeaddim || dstate > kMaxDstate)
        return fail(SSD_ERR_UNSUPPORTED, "the backward handles headdim <= %d and dstate <= %d (got %d, %d)",
                    kBwdMaxHeaddim, kMaxDstate, headdim, dstate);
    if (nheads > 65535 || batch > 65535)
        return fail(SSD_ERR_UNSUPPORTED, "nheads and batch must each be <= 65535");
    p.batch = batch;
    p.seqlen = seqlen;
    p.nheads = nheads;
    p.headdim = headdim;
    p.ngroups = ngroups;
    p.dstate = dstate;
    p.dtype = dtype;
    return SSD_OK;
}

ssd_status_t ssd_bwd(const void *x, const float *dt, const float *A, const void *B, const void *C, const float *D,
                     const float *init_state, const void *dy, const float *dfinal_state, float *dx, float *ddt,
                     float *dA, float *dB, float *dC, float *dD, float *dinit_state, int batch, int seqlen,
                     int nheads, int headdim, int ngroups, int dstate, ssd_dtype_t dtype, void *stream)
{
    BwdProblem p;
    ssd_status_t st = make_bwd_problem(p, batch, seqlen, nheads, headdim, ngroups, dstate, dtype);
    if (st != SSD_OK) return st;
    if (!x || !dt || !A || !B || !C || !dy || !dx || !ddt || !dA || !dB || !dC)
        return fail(SSD_ERR_INVALID_ARG, "x, dt, A, B, C, dy, dx, ddt, dA, dB and dC must be non-NULL");
    const size_t el = dtype == SSD_DTYPE_BF16 ? 2 : 4;
    if (!aligned(x, el) || !aligned(B, el) || !aligned(C, el) || !aligned(dy, el))
        return fail(SSD_ERR_INVALID_ARG, "x, B, C and dy must be aligned to their element size");
    const void *f32[] = {dt, A, D, init_state, dfinal_state, dx, ddt, dA, dB, dC, dD, dinit_state};
    for (const void *q : f32)
        if (q && !aligned(q, 4)) return fail(SSD_ERR_INVALID_ARG, "fp32 tensors must be 4-byte aligned");
    p.x = x;
    p.dt = dt;
    p.A = A;
    p.B = B;
    p.C = C;
    p.D = D;
    p.init_state = init_state;
    p.dy = dy;
    p.dfinal = dfinal_state;
    p.dx = dx;
    p.ddt = ddt;
    p.dA = dA;
    p.dB = dB;
    p.dC = dC;
    p.dD = dD;
    p.dinit = dinit_state;
    p.err_word = device_error_word();
    if (!p.err_word) return fail(SSD_ERR_CUDA, "cannot resolve the device error word");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t need = bwd_workspace_bytes(p);
    void *ws = nullptr;
    cudaError_t e = cudaMallocAsync(&ws, need, s);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(e == cudaErrorMemoryAllocation ? SSD_ERR_NO_MEMORY : SSD_ERR_CUDA,
                    "workspace allocation of %zu bytes failed: %s", need, cudaGetErrorString(e));
    }
    profile_forward_begin();
    e = launch_bwd(p, ws, s);
    const cudaError_t ef = cudaFreeAsync(ws, s);
    if (e != cudaSuccess) return fail(SSD_ERR_CUDA, "backward launch failed: %s", cudaGetErrorString(e));
    if (ef != cudaSuccess) return fail(SSD_ERR_CUDA, "workspace release failed: %s", cudaGetErrorString(ef));
    return ok();
}

int ssd_bwd_kernels(int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate, ssd_dtype_t dtype,
                    char *names, size_t names_len)
{
    BwdProblem p;
    if (make_bwd_problem(p, batch, seqlen, nheads, headdim, ngroups, dstate, dtype) != SSD_OK) return -1;
    if (names && names_len) snprintf(names, names_len, "%s", bwd_kernel_names(p));
    return bwd_kernel_count(p);
}

ssd_status_t ssd_bwd_workspace_size(int batch, int seqlen, int nheads, int headdim, int ngroups, int dstate,
                                    ssd_dtype_t dtype, size_t *bytes)
{
    if (!bytes) return fail(SSD_ERR_INVALID_ARG, "bytes must be non-NULL");
    BwdProblem p;
    ssd_status_t st = make_bwd_problem(p, batch, seqlen, nheads, headdim, ngroups, dstate, dtype);
    if (st != SSD_OK) return st;
    *bytes = bwd_workspace_bytes(p);
    return ok();
}

ssd_status_t ssd_test_set_fault(unsigned long long wait_limit_ns, long long withhold_unit)
{
    if (withhold_unit < -1) return fail(SSD_ERR_INVALID_ARG, "withhold_unit must be -1 or a unit index");
    t_wait_ns = wait_limit_ns;
    t_withhold = withhold_unit;
    return ok();
}

ssd_status_t ssd_check_device_status(void *stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(SSD_ERR_CUDA, "stream error: %s", cudaGetErrorString(e));
    unsigned int word = 0;
    const unsigned int zero = 0;
    e = cudaMemcpyFromSymbol(&word, g_device_error, sizeof word);
    if (e == cudaSuccess && word) e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
    if (e != cudaSuccess) return fail(SSD_ERR_CUDA, "reading the device error word failed: %s",
                                      cudaGetErrorString(e));
    if (word & kDevErrTimeout) return fail(SSD_ERR_TIMEOUT, "a bounded device-side wait gave up (word 0x%x)", word);
    if (word & kDevErrBounds) return fail(SSD_ERR_INVALID_ARG, "a kernel-side check failed (word 0x%x)", word);
    return ok();
}

const char *ssd_status_string(ssd_status_t status)
{
    switch (status) {
    case SSD_OK: return "SSD_OK";
    case SSD_ERR_INVALID_ARG: return "SSD_ERR_INVALID_ARG: invalid argument";
    case SSD_ERR_UNSUPPORTED: return "SSD_ERR_UNSUPPORTED: outside the sizes this build handles";
    case SSD_ERR_CUDA: return "SSD_ERR_CUDA: CUDA runtime error";
    case SSD_ERR_NO_MEMORY: return "SSD_ERR_NO_MEMORY: allocation failed";
    case SSD_ERR_TIMEOUT: return "SSD_ERR_TIMEOUT: bounded device-side wait gave up";
    }
    return "unknown ssd_status_t";
}

const char *ssd_last_error_detail(void) { return g_detail; }

const char *ssd_version(void) { return "libssd 0.1 (sm_103a)"; }

}  // extern "C"
