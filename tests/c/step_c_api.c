/*
 * step_c_api.c -- the C ABI used from plain C: one tiny decoding step (fp32,
 * d = 64, V = 1000, K = 3 heads, s = (2,2,2), 14 tree nodes, one attention
 * head of dim 64 over 32 prefix slots) issued as the four separate calls and
 * through the step executor (stream and graph mode, inputs copied from
 * page-locked host memory, results written to page-locked host memory),
 * compared bit for bit.  Prints "ok" and exits 0 on success.
 *
 * Inputs are arbitrary test data from a small linear congruential
 * generator: the check is that the paths agree, not what they compute (the
 * Python parity tests compare the calls with the oracle).
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "medusa.h"

enum { B = 1, D = 64, V = 1000, K = 3, S = 2, N = 14, R = N + 1, H = 1, DH = 64, P = 32 };

#define CK(x)                                                                    \
    do {                                                                         \
        cudaError_t e_ = (x);                                                    \
        if (e_ != cudaSuccess) {                                                 \
            fprintf(stderr, "%s:%d %s\n", __FILE__, __LINE__, cudaGetErrorString(e_)); \
            exit(2);                                                             \
        }                                                                        \
    } while (0)
#define MK(x)                                                                    \
    do {                                                                         \
        medusa_status s_ = (x);                                                  \
        if (s_ != MEDUSA_OK) {                                                   \
            fprintf(stderr, "%s:%d %s: %s\n", __FILE__, __LINE__,                \
                    medusa_status_string(s_), medusa_last_error());              \
            exit(3);                                                             \
        }                                                                        \
    } while (0)

static uint64_t lcg = 0x9e3779b97f4a7c15ull;
static float next_uniform(void) { /* in [-1, 1) */
    lcg = lcg * 6364136223846793005ull + 1442695040888963407ull;
    return (float)((lcg >> 40) & 0xffffff) / 8388608.0f - 1.0f;
}
static void fill(float *x, size_t n, float scale) {
    for (size_t i = 0; i < n; ++i) x[i] = scale * next_uniform();
}
static void *dalloc(size_t bytes) {
    void *p = NULL;
    CK(cudaMalloc(&p, bytes));
    CK(cudaMemset(p, 0, bytes));
    return p;
}
static void *halloc(size_t bytes) {
    void *p = NULL;
    CK(cudaHostAlloc(&p, bytes, cudaHostAllocDefault));
    memset(p, 0, bytes);
    return p;
}

/* everything the step writes, copied to the host for comparison */
struct Results {
    int32_t ids[B * K * S], tokens[B * R], parent[B * R], depth[B * R], pos_id[B * R];
    uint64_t anc[B * R];
    float logp[B * K * S], out[B * R * H * DH];
    int32_t accept_len[B], path[B * (K + 1)], path_tokens[B * (K + 1)], next_token[B];
};

int main(void) {
    const int32_t s_host[K] = {S, S, S};
    const size_t hb = sizeof(float) * B * D, qb = sizeof(float) * B * R * H * DH,
                 lb = sizeof(float) * B * R * V, cb = sizeof(float) * (P + R) * H * DH;
    /* weights and caches: device-resident, filled once */
    float *hW1 = malloc(sizeof(float) * K * D * D), *hW2 = malloc(sizeof(float) * K * V * D);
    float *hk = malloc(cb), *hv = malloc(cb);
    fill(hW1, (size_t)K * D * D, 0.05f);
    fill(hW2, (size_t)K * V * D, 0.2f);
    fill(hk, cb / sizeof(float), 1.0f);
    fill(hv, cb / sizeof(float), 1.0f);
    float *W1 = dalloc(sizeof(float) * K * D * D), *W2 = dalloc(sizeof(float) * K * V * D);
    float *kc = dalloc(cb), *vc = dalloc(cb);
    CK(cudaMemcpy(W1, hW1, sizeof(float) * K * D * D, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(W2, hW2, sizeof(float) * K * V * D, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(kc, hk, cb, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(vc, hv, cb, cudaMemcpyHostToDevice));
    void **kp = dalloc(sizeof(void *)), **vp = dalloc(sizeof(void *));
    CK(cudaMemcpy(kp, &kc, sizeof(void *), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(vp, &vc, sizeof(void *), cudaMemcpyHostToDevice));
    int32_t *prefix = dalloc(sizeof(int32_t) * B);
    const int32_t hp = P;
    CK(cudaMemcpy(prefix, &hp, sizeof hp, cudaMemcpyHostToDevice));

    /* the step's inputs: pinned host sources and their device homes */
    float *h_host = halloc(hb), *q_host = halloc(qb), *logits_host = halloc(lb);
    int32_t *root_host = halloc(sizeof(int32_t) * B);
    float *h = dalloc(hb), *q = dalloc(qb), *logits = dalloc(lb);
    int32_t *root = dalloc(sizeof(int32_t) * B);

    /* outputs and scratch */
    int32_t *ids = dalloc(sizeof(int32_t) * B * K * S);
    float *logp = dalloc(sizeof(float) * B * K * S);
    int32_t *tokens = dalloc(sizeof(int32_t) * B * R), *parent = dalloc(sizeof(int32_t) * B * R);
    int32_t *depth = dalloc(sizeof(int32_t) * B * R), *pos_id = dalloc(sizeof(int32_t) * B * R);
    uint64_t *anc = dalloc(sizeof(uint64_t) * B * R);
    int32_t *paths = dalloc(sizeof(int32_t) * B * N * (K + 1)), *n_leaf = dalloc(sizeof(int32_t) * B);
    float *out = dalloc(qb);
    int32_t *acc_len = halloc(sizeof(int32_t) * B), *path = halloc(sizeof(int32_t) * B * (K + 1));
    int32_t *path_tok = halloc(sizeof(int32_t) * B * (K + 1)), *next = halloc(sizeof(int32_t) * B);
    size_t wsb = medusa_heads_workspace_size(B, K, D, V, S);
    size_t t = medusa_build_tree_workspace_size(B, K, S, N);
    if (t > wsb) wsb = t;
    t = medusa_tree_attention_workspace_size(MEDUSA_F32, B, R, H, DH, P);
    if (t > wsb) wsb = t;
    t = medusa_posterior_workspace_size(B, R);
    if (t > wsb) wsb = t;
    void *ws = dalloc(wsb);
    const float scale = 1.0f / sqrtf((float)DH);
    cudaStream_t st;
    CK(cudaStreamCreate(&st));

    struct Results ref, got;
    memset(&ref, 0, sizeof ref);  /* padding compares equal too */
    memset(&got, 0, sizeof got);
#define COLLECT(r)                                                                       \
    do {                                                                                 \
        CK(cudaStreamSynchronize(st));                                                   \
        CK(cudaMemcpy((r).ids, ids, sizeof (r).ids, cudaMemcpyDeviceToHost));            \
        CK(cudaMemcpy((r).logp, logp, sizeof (r).logp, cudaMemcpyDeviceToHost));         \
        CK(cudaMemcpy((r).tokens, tokens, sizeof (r).tokens, cudaMemcpyDeviceToHost));   \
        CK(cudaMemcpy((r).parent, parent, sizeof (r).parent, cudaMemcpyDeviceToHost));   \
        CK(cudaMemcpy((r).depth, depth, sizeof (r).depth, cudaMemcpyDeviceToHost));      \
        CK(cudaMemcpy((r).pos_id, pos_id, sizeof (r).pos_id, cudaMemcpyDeviceToHost));   \
        CK(cudaMemcpy((r).anc, anc, sizeof (r).anc, cudaMemcpyDeviceToHost));            \
        CK(cudaMemcpy((r).out, out, sizeof (r).out, cudaMemcpyDeviceToHost));            \
        memcpy((r).accept_len, acc_len, sizeof (r).accept_len);                          \
        memcpy((r).path, path, sizeof (r).path);                                         \
        memcpy((r).path_tokens, path_tok, sizeof (r).path_tokens);                       \
        memcpy((r).next_token, next, sizeof (r).next_token);                             \
    } while (0)

    medusa_copy early[2] = {{h, h_host, hb}, {root, root_host, sizeof(int32_t) * B}};
    medusa_copy late[2] = {{q, q_host, qb}, {logits, logits_host, lb}};
    medusa_step_desc desc;
    memset(&desc, 0, sizeof desc);
    desc.early = early; desc.n_early = 2; desc.late = late; desc.n_late = 2;
    desc.dtype = MEDUSA_F32;
    desc.h = h; desc.W1 = W1; desc.b1 = NULL; desc.W2 = W2;
    desc.B = B; desc.d = D; desc.V = V; desc.K = K; desc.top_s = S;
    desc.topk_ids = ids; desc.topk_logp = logp;
    desc.root = root; desc.s_host = s_host; desc.n = N; desc.prefix_len = prefix;
    desc.tokens = tokens; desc.parent = parent; desc.depth = depth; desc.pos_id = pos_id;
    desc.anc_mask = anc; desc.paths = paths; desc.n_leaf = n_leaf;
    desc.q = q; desc.k_cache = (const void *const *)kp; desc.v_cache = (const void *const *)vp;
    desc.P_max = P; desc.H = H; desc.dh = DH; desc.scale = scale; desc.attn_out = out;
    desc.logits = logits; desc.mode = MEDUSA_TYPICAL; desc.eps = 0.09f; desc.delta = 0.3f;
    desc.temperature = 1.0f;
    desc.accept_len = acc_len; desc.path = path; desc.path_tokens = path_tok;
    desc.next_token = next; desc.accept = NULL; desc.new_prefix_len = NULL;
    desc.ws = ws; desc.ws_bytes = wsb;
    if (medusa_step_desc_size() != sizeof(medusa_step_desc)) {
        fprintf(stderr, "descriptor size differs from the library's\n");
        return 4;
    }
    medusa_step_exec *ex_stream = NULL, *ex_graph = NULL;
    MK(medusa_step_create(&desc, &ex_stream));
    desc.flags = MEDUSA_STEP_GRAPH;
    MK(medusa_step_create(&desc, &ex_graph));

    for (int rep = 0; rep < 3; ++rep) {
        fill(h_host, hb / sizeof(float), 1.0f);
        root_host[0] = (int32_t)((lcg >> 33) % V);
        fill(q_host, qb / sizeof(float), 1.0f);
        fill(logits_host, lb / sizeof(float), 3.0f);

        /* the separate calls (the copies first, by hand) */
        CK(cudaMemcpyAsync(h, h_host, hb, cudaMemcpyHostToDevice, st));
        CK(cudaMemcpyAsync(root, root_host, sizeof(int32_t) * B, cudaMemcpyHostToDevice, st));
        CK(cudaMemcpyAsync(q, q_host, qb, cudaMemcpyHostToDevice, st));
        CK(cudaMemcpyAsync(logits, logits_host, lb, cudaMemcpyHostToDevice, st));
        MK(medusa_heads(MEDUSA_F32, h, W1, NULL, W2, B, D, V, K, S, ids, logp, ws, wsb, st));
        MK(medusa_build_tree(root, ids, logp, B, K, s_host, S, N, prefix, tokens, parent, depth,
                             pos_id, anc, paths, n_leaf, ws, wsb, st));
        MK(medusa_tree_attention(MEDUSA_F32, q, (const void *const *)kp,
                                 (const void *const *)vp, prefix, P, anc, B, R, H, DH, scale, out,
                                 ws, wsb, st));
        MK(medusa_evaluate_posterior(MEDUSA_F32, logits, tokens, parent, depth, B, R, V, K,
                                     MEDUSA_TYPICAL, 0.09f, 0.3f, 1.0f, acc_len, path, path_tok,
                                     next, NULL, ws, wsb, st));
        COLLECT(ref);
        if (ref.tokens[0] != root_host[0]) {
            fprintf(stderr, "rep %d: the tree's root is not the input root\n", rep);
            return 5;
        }
        medusa_step_exec *exs[2] = {ex_stream, ex_graph};
        for (int m = 0; m < 2; ++m) {
            CK(cudaMemset(out, 0, qb));
            CK(cudaMemset(tokens, 0, sizeof(int32_t) * B * R));
            memset(next, 0xff, sizeof(int32_t) * B);
            if (rep == 2) { /* the wait on its own */
                MK(medusa_step_run(exs[m], st, 0));
                MK(medusa_step_wait(exs[m], st));
            } else {
                MK(medusa_step_run(exs[m], st, 1));
            }
            COLLECT(got);
            if (memcmp(&ref, &got, sizeof ref) != 0) {
                fprintf(stderr, "rep %d: the %s executor differs from the calls\n", rep,
                        m ? "graph-mode" : "stream-mode");
                return 6;
            }
        }
    }
    int32_t status = -1;
    MK(medusa_read_device_status(ws, &status, st));
    if (status != MEDUSA_DEV_OK) {
        fprintf(stderr, "device status %d\n", status);
        return 7;
    }
    medusa_step_destroy(ex_graph);
    medusa_step_destroy(ex_stream);
    CK(cudaStreamDestroy(st));
    printf("ok\n");
    return 0;
}
