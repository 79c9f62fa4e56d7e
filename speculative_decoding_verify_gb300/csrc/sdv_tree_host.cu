// sdv_tree_host.cu - the accepted path of a greedy draft tree as node indices, on the host: the
// rows sd_kv_commit keeps ("How Kinetic is fast", section "Why the output does not change": a
// node is kept when its parent is and its token is the parent's top token; "Speculative Decoding
// with Open-Weights Models", section "Engineering the Architecture: KV Cache Synchronization").
// The same rule as sd_accept_greedy with a parent array; the caller copies the few int32 it
// needs (argmax, tokens, parent) to the host, as it already does for the accepted tokens.
#include "sdverify.h"

extern "C" {

int32_t sd_tree_path(const int32_t *argmax, const int32_t *tokens, const int32_t *parent, int32_t M, int32_t *path) {
    if (!argmax || !tokens || !parent || !path || M < 1 || M > 16 || parent[0] != -1) return -1;
    int32_t depth[16] = {0};
    bool ok[16] = {true};
    int32_t best = 0;
    for (int32_t i = 1; i < M; ++i) {
        const int32_t p = parent[i];
        if (p < 0 || p >= i) return -1;
        depth[i] = depth[p] + 1;
        ok[i] = ok[p] && tokens[i] == argmax[p];
        if (ok[i] && depth[i] > depth[best]) best = i;  // the deepest, lowest index among equals
    }
    for (int32_t i = best, j = depth[best]; j >= 0; i = parent[i], --j) path[j] = i;
    return depth[best] + 1;
}

}  // extern "C"
