// step.cu -- the step executor: one host call issues a whole decoding step.
//
// "Medusa: Faster LLM text generation", Introduction, and "Medusa 深读" §3-§6:
// a step is heads -> candidate tree -> tree attention -> posterior (and the
// commit).  The executor issues that sequence through the public calls of
// this library, together with the step's input copies from page-locked host
// memory: the heads' inputs first on the caller's stream, the attention's and
// the posterior's on a side stream while the heads stream the weights,
// joined before the attention.  Issued from here, the step's launches leave
// the host a few microseconds apart, far ahead of the GPU, and each kernel
// keeps its programmatic-dependent-launch overlap with the one before it;
// in graph mode the sequence is captured once and each run is one graph
// launch.  When the results are page-locked host memory, the wait for a
// step polls completion words that the posterior's last kernel raises after
// its writes, which land a few microseconds before the stream would report
// the step complete.
#include <chrono>
#include <cstring>
#include <new>

#include "launch.h"

struct medusa_step_exec {
    medusa_step_desc desc;
    medusa_copy early[MEDUSA_STEP_MAX_COPIES];
    medusa_copy late[MEDUSA_STEP_MAX_COPIES];
    // each copy's direction, resolved once at create (a copy of kind
    // cudaMemcpyDefault would have its pointers looked up at every issue)
    cudaMemcpyKind early_kind[MEDUSA_STEP_MAX_COPIES];
    cudaMemcpyKind late_kind[MEDUSA_STEP_MAX_COPIES];
    int32_t s_host[MEDUSA_MAX_HEADS];
    cudaStream_t side;
    cudaEvent_t fork, join;
    // graph mode: the sequence captured once, and the kernels it launches
    cudaGraphExec_t graph;
    uint64_t graph_launches;
    // with page-locked results: one completion word per sequence, raised by
    // the posterior's last kernel once per run, and the runs issued
    uint32_t *done;
    uint32_t runs;
};

namespace {

using medusa::set_last_error;

medusa_status invalid(const char *what) {
    set_last_error("medusa_step_create: %s", what);
    return MEDUSA_ERR_INVALID_ARG;
}

medusa_status cuda_error(cudaError_t e, const char *where) {
    set_last_error("%s: %s", where, cudaGetErrorString(e));
    return MEDUSA_ERR_CUDA;
}

medusa_status check_copies(const medusa_copy *c, int32_t n, const char *which) {
    if (n < 0 || n > MEDUSA_STEP_MAX_COPIES) {
        set_last_error("medusa_step_create: %s copy count %d outside 0..%d", which, n,
                       MEDUSA_STEP_MAX_COPIES);
        return MEDUSA_ERR_INVALID_ARG;
    }
    if (n > 0 && !c) return invalid(which[0] == 'e' ? "early copy list is NULL"
                                                    : "late copy list is NULL");
    for (int32_t i = 0; i < n; ++i)
        if (!c[i].dst || !c[i].src || c[i].bytes == 0) {
            set_last_error("medusa_step_create: %s copy %d has a NULL pointer or no bytes", which,
                           i);
            return MEDUSA_ERR_INVALID_ARG;
        }
    return MEDUSA_OK;
}

// The descriptor's structure; shapes, alignments and workspace sizes are
// checked by each call when the step runs.
medusa_status check_desc(const medusa_step_desc &d) {
    if (medusa_status s = check_copies(d.early, d.n_early, "early")) return s;
    if (medusa_status s = check_copies(d.late, d.n_late, "late")) return s;
    if (d.dtype != MEDUSA_F32 && d.dtype != MEDUSA_BF16) return invalid("unknown dtype");
    if (d.B < 1 || d.B > MEDUSA_MAX_BATCH) return invalid("B outside 1..8");
    if (d.K < 1 || d.K > MEDUSA_MAX_HEADS) return invalid("K outside 1..8");
    if (d.top_s < 1 || d.top_s > MEDUSA_MAX_TOP_S) return invalid("top_s outside 1..16");
    if (d.n < 1 || d.n + 1 > MEDUSA_MAX_TREE_ROWS) return invalid("n + 1 outside 2..256");
    if (d.d < 1 || d.V < 1 || d.H < 1 || d.dh < 1 || d.P_max < 0)
        return invalid("d, V, H, dh must be positive and P_max non-negative");
    if (d.flags & ~MEDUSA_STEP_GRAPH) return invalid("unknown flags");
    if (!d.s_host) return invalid("s_host is NULL");
    for (int k = 0; k < d.K; ++k)
        if (d.s_host[k] < 1 || d.s_host[k] > d.top_s) return invalid("s_host[k] outside 1..top_s");
    const void *need[] = {d.h, d.W1, d.W2, d.topk_ids, d.topk_logp, d.root, d.prefix_len,
                          d.tokens, d.parent, d.depth, d.pos_id, d.anc_mask, d.paths, d.n_leaf,
                          d.q, d.k_cache, d.v_cache, d.attn_out, d.logits, d.accept_len, d.path,
                          d.path_tokens, d.next_token, d.ws};
    for (const void *p : need)
        if (!p) return invalid("a required buffer is NULL (only b1, accept, new_prefix_len "
                               "may be)");
    return MEDUSA_OK;
}

// The direction of each copy: the destination must be device memory, the
// source page-locked host memory or device memory.
medusa_status resolve_kinds(const medusa_copy *c, int32_t n, cudaMemcpyKind *kind,
                            const char *which) {
    for (int32_t i = 0; i < n; ++i) {
        cudaPointerAttributes a{}, b{};
        cudaError_t e = cudaPointerGetAttributes(&a, c[i].dst);
        if (!e) e = cudaPointerGetAttributes(&b, c[i].src);
        if (e) {
            cudaGetLastError();
            set_last_error("medusa_step_create: %s copy %d: %s", which, i, cudaGetErrorString(e));
            return MEDUSA_ERR_INVALID_ARG;
        }
        if (a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) {
            set_last_error("medusa_step_create: %s copy %d: destination is not device memory",
                           which, i);
            return MEDUSA_ERR_INVALID_ARG;
        }
        if (b.type == cudaMemoryTypeHost) {
            kind[i] = cudaMemcpyHostToDevice;
        } else if (b.type == cudaMemoryTypeDevice || b.type == cudaMemoryTypeManaged) {
            kind[i] = cudaMemcpyDeviceToDevice;
        } else {
            set_last_error("medusa_step_create: %s copy %d: source is neither page-locked host "
                           "memory nor device memory", which, i);
            return MEDUSA_ERR_INVALID_ARG;
        }
    }
    return MEDUSA_OK;
}

// The step's sequence on `st` (the caller's stream, or the capture stream).
medusa_status issue_step(medusa_step_exec *ex, cudaStream_t st) {
    const medusa_step_desc &d = ex->desc;
    const int R = d.n + 1;
    cudaError_t e;
    // the side stream's copies overwrite buffers that earlier work on
    // `stream` (the previous step's attention and posterior) reads
    if (d.n_late > 0 && (e = cudaEventRecord(ex->fork, st)))
        return cuda_error(e, "medusa_step (fork)");
    for (int i = 0; i < d.n_early; ++i)
        if ((e = cudaMemcpyAsync(d.early[i].dst, d.early[i].src, d.early[i].bytes,
                                 ex->early_kind[i], st)))
            return cuda_error(e, "medusa_step (early copy)");
    if (medusa_status s = medusa_heads(d.dtype, d.h, d.W1, d.b1, d.W2, d.B, d.d, d.V, d.K,
                                       d.top_s, d.topk_ids, d.topk_logp, d.ws, d.ws_bytes, st))
        return s;
    if (d.n_late > 0) {
        if ((e = cudaStreamWaitEvent(ex->side, ex->fork, 0)))
            return cuda_error(e, "medusa_step (side wait)");
        for (int i = 0; i < d.n_late; ++i)
            if ((e = cudaMemcpyAsync(d.late[i].dst, d.late[i].src, d.late[i].bytes,
                                     ex->late_kind[i], ex->side)))
                return cuda_error(e, "medusa_step (late copy)");
        if ((e = cudaEventRecord(ex->join, ex->side)))
            return cuda_error(e, "medusa_step (join)");
    }
    if (medusa_status s = medusa_build_tree(d.root, d.topk_ids, d.topk_logp, d.B, d.K, d.s_host,
                                            d.top_s, d.n, d.prefix_len, d.tokens, d.parent,
                                            d.depth, d.pos_id, d.anc_mask, d.paths, d.n_leaf,
                                            d.ws, d.ws_bytes, st))
        return s;
    if (d.n_late > 0 && (e = cudaStreamWaitEvent(st, ex->join, 0)))
        return cuda_error(e, "medusa_step (join wait)");
    if (medusa_status s = medusa_tree_attention(d.dtype, d.q, d.k_cache, d.v_cache, d.prefix_len,
                                                d.P_max, d.anc_mask, d.B, R, d.H, d.dh, d.scale,
                                                d.attn_out, d.ws, d.ws_bytes, st))
        return s;
    const bool commit = d.new_prefix_len != nullptr;
    return medusa::evaluate_posterior_signalled(
        d.dtype, d.logits, d.tokens, d.parent, d.depth, d.B, R, d.V, d.K, d.mode, d.eps, d.delta,
        d.temperature, d.accept_len, d.path, d.path_tokens, d.next_token, d.accept,
        commit ? const_cast<void *const *>(d.k_cache) : nullptr,
        commit ? const_cast<void *const *>(d.v_cache) : nullptr, commit ? d.prefix_len : nullptr,
        d.H, d.dh, d.new_prefix_len, d.ws, d.ws_bytes, st, ex->done);
}

// Wait for run number `runs`: with completion words, until every sequence's
// word has reached it (the results are then in host memory), with a time
// limit after which the stream is synchronised instead; otherwise the
// stream.
medusa_status wait_step(medusa_step_exec *ex, cudaStream_t st) {
    if (ex->done) {
        const volatile uint32_t *w = ex->done;
        const auto t0 = std::chrono::steady_clock::now();
        for (uint32_t polls = 1;; ++polls) {
            bool all = true;
            for (int b = 0; b < ex->desc.B && all; ++b)
                all = static_cast<int32_t>(w[b] - ex->runs) >= 0;
            if (all) return MEDUSA_OK;
            if ((polls & 1023u) == 0 &&
                std::chrono::steady_clock::now() - t0 > std::chrono::milliseconds(20))
                break;
        }
    }
    cudaError_t e = cudaStreamSynchronize(st);
    if (e) return cuda_error(e, "medusa_step_run (synchronize)");
    if (ex->done) ex->runs = ex->done[0];  // realign after the fallback
    return MEDUSA_OK;
}

// Graph mode: the sequence issued once on a capture stream of its own (the
// side stream joins the capture through the fork event and leaves it through
// the join), then instantiated.  Relaxed capture, so that the calls' host
// checks (pointer attributes) are allowed while capturing.
medusa_status capture_step(medusa_step_exec *ex) {
    cudaStream_t cap;
    cudaError_t e = cudaStreamCreateWithFlags(&cap, cudaStreamNonBlocking);
    if (e) return cuda_error(e, "medusa_step_create (capture stream)");
    const uint64_t launches0 = medusa_launch_count();
    if ((e = cudaStreamBeginCapture(cap, cudaStreamCaptureModeRelaxed))) {
        cudaStreamDestroy(cap);
        return cuda_error(e, "medusa_step_create (begin capture)");
    }
    medusa_status s = issue_step(ex, cap);
    cudaGraph_t graph = nullptr;
    e = cudaStreamEndCapture(cap, &graph);  // always leaves capture mode
    if (!s && e) s = cuda_error(e, "medusa_step_create (end capture)");
    if (!s && (e = cudaGraphInstantiate(&ex->graph, graph, 0))) {
        ex->graph = nullptr;
        s = cuda_error(e, "medusa_step_create (instantiate)");
    }
    if (graph) cudaGraphDestroy(graph);
    cudaStreamDestroy(cap);
    if (s) cudaGetLastError();  // a failed capture leaves no error for later calls
    // the kernels one replay launches (the process-wide counter: launches
    // by other threads during the capture would be counted too)
    ex->graph_launches = medusa_launch_count() - launches0;
    return s;
}

}  // namespace

extern "C" {

size_t medusa_step_desc_size(void) { return sizeof(medusa_step_desc); }

medusa_status medusa_step_create(const medusa_step_desc *desc, medusa_step_exec **exec_out) {
    if (!desc || !exec_out) return invalid("NULL descriptor or output pointer");
    *exec_out = nullptr;
    if (medusa_status s = check_desc(*desc)) return s;
    medusa_step_exec *ex = new (std::nothrow) medusa_step_exec();
    if (!ex) {
        set_last_error("medusa_step_create: out of host memory");
        return MEDUSA_ERR_INVALID_ARG;
    }
    ex->desc = *desc;
    if (desc->n_early) std::memcpy(ex->early, desc->early, sizeof(medusa_copy) * desc->n_early);
    if (desc->n_late) std::memcpy(ex->late, desc->late, sizeof(medusa_copy) * desc->n_late);
    std::memcpy(ex->s_host, desc->s_host, sizeof(int32_t) * desc->K);
    ex->desc.early = ex->early;
    ex->desc.late = ex->late;
    ex->desc.s_host = ex->s_host;
    medusa_status sk = resolve_kinds(ex->early, desc->n_early, ex->early_kind, "early");
    if (!sk) sk = resolve_kinds(ex->late, desc->n_late, ex->late_kind, "late");
    if (sk) {
        delete ex;
        return sk;
    }
    cudaError_t e = cudaStreamCreateWithFlags(&ex->side, cudaStreamNonBlocking);
    if (e) {
        delete ex;
        return cuda_error(e, "medusa_step_create (side stream)");
    }
    // results in page-locked host memory: completion words beside them
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, desc->accept_len) == cudaSuccess &&
        at.type == cudaMemoryTypeHost) {
        void *p = nullptr;
        void *dp = nullptr;
        if (cudaHostAlloc(&p, sizeof(uint32_t) * desc->B, cudaHostAllocMapped) == cudaSuccess) {
            if (cudaHostGetDevicePointer(&dp, p, 0) == cudaSuccess && dp == p) {
                std::memset(p, 0, sizeof(uint32_t) * desc->B);
                ex->done = static_cast<uint32_t *>(p);
            } else {
                cudaFreeHost(p);
            }
        }
    }
    cudaGetLastError();  // the probes above leave no error behind
    e = cudaEventCreateWithFlags(&ex->fork, cudaEventDisableTiming);
    if (!e) {
        e = cudaEventCreateWithFlags(&ex->join, cudaEventDisableTiming);
        if (e) cudaEventDestroy(ex->fork);
    }
    if (e) {
        cudaStreamDestroy(ex->side);
        if (ex->done) cudaFreeHost(ex->done);
        delete ex;
        return cuda_error(e, "medusa_step_create (events)");
    }
    if (desc->flags & MEDUSA_STEP_GRAPH) {
        if (medusa_status s = capture_step(ex)) {
            medusa_step_destroy(ex);
            return s;
        }
    }
    *exec_out = ex;
    return MEDUSA_OK;
}

medusa_status medusa_step_run(medusa_step_exec *ex, medusa_stream stream, int synchronize) {
    const medusa::NvtxRange range("medusa_step_run");
    if (!ex) {
        set_last_error("medusa_step_run: NULL executor");
        return MEDUSA_ERR_INVALID_ARG;
    }
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (ex->graph) {
        if ((e = cudaGraphLaunch(ex->graph, st))) return cuda_error(e, "medusa_step_run (graph)");
        for (uint64_t i = 0; i < ex->graph_launches; ++i) medusa::note_launch();
    } else if (medusa_status s = issue_step(ex, st)) {
        return s;
    }
    ++ex->runs;  // the posterior was issued: its words will reach this count
    return synchronize ? wait_step(ex, st) : MEDUSA_OK;
}

medusa_status medusa_step_wait(medusa_step_exec *ex, medusa_stream stream) {
    if (!ex) {
        set_last_error("medusa_step_wait: NULL executor");
        return MEDUSA_ERR_INVALID_ARG;
    }
    return wait_step(ex, static_cast<cudaStream_t>(stream));
}

void medusa_step_destroy(medusa_step_exec *ex) {
    if (!ex) return;
    // each releases its resources once the work it carries has completed
    if (ex->graph) cudaGraphExecDestroy(ex->graph);
    if (ex->done) {
        cudaStreamSynchronize(ex->side);
        cudaFreeHost(ex->done);  // synchronises the device first
    }
    cudaEventDestroy(ex->join);
    cudaEventDestroy(ex->fork);
    cudaStreamDestroy(ex->side);
    delete ex;
}

}  // extern "C"
