/*
 * tt_graph.h -- the generic tensor graph of a context: tensors bump-allocated
 * from the context's arena, each recording the op and the inputs that made
 * it, evaluated forward and differentiated backward on the device.
 *
 * Pages the calls follow (cited by title and section):
 *  - tinytorch ("不用PyTorch，一个头文件就能训练GPT-2：Arena内存池+自动微分的C++实现"):
 *    三.1 NewTensor cuts each tensor (value and gradient) out of the arena and
 *    Reset releases all of them at once; 三.2 a tensor records its op and its
 *    inputs; 三.3 Forward evaluates the inputs first, Backward passes the
 *    gradient back with +=, MatMul is C = A B with B [K, N]; 三.4 GELU;
 *    三.5 Softmax and CrossEntropy, and the gradient probs - onehot when the
 *    two meet; 八.5 the example: the graph is built once and Forward,
 *    ZeroGrad, Backward and an SGD update run every step.
 *  - microcrad: Values 的工作原理 (c = a * b gives dc/da = b, dc/db = a),
 *    反向传播 (a topological order, the seed gradient 1), 关于 magic 字段的说明
 *    (handles are checked before use).
 *
 * Conventions (in addition to those of tt.h):
 *  - A node handle is an int32 >= 0.  Calls that make a node return the
 *    handle, or a negative tt_status on failure (message in tt_last_error).
 *  - Nodes live until tt_ctx_reset, which also releases their memory; a
 *    handle made before a reset is stale afterwards (TT_ERR_STALE), and so is
 *    a handle of another context.
 *  - Values are float32 (TT_NODE_F32) or int32 labels (TT_NODE_I32, no
 *    gradient).  Every f32 node has a gradient buffer of its own shape,
 *    zeroed when the node is made.
 *  - Evaluation order is the order in which nodes were made, which is a
 *    topological order because a node's inputs exist before it.
 *  - Every kernel reduces in a fixed order: results are deterministic.
 */
#ifndef TT_GRAPH_H
#define TT_GRAPH_H

#include "tt.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t tt_node;

typedef enum { TT_NODE_F32 = 0, TT_NODE_I32 = 1 } tt_node_type;

/* A leaf tensor of ndim (1..4) dimensions, values zero (tinytorch 三.1
 * NewTensor).  TT_ERR_ARG for a bad shape or type, TT_ERR_ARENA_OOM when the
 * arena cannot hold its value and gradient. */
tt_node tt_node_new(tt_ctx* ctx, int ndim, const int* shape, tt_node_type type);

/* C = A B for A [M, K] and B [K, N] (tinytorch 三.3).  Both f32 2-D with
 * matching K, else TT_ERR_ARG. */
tt_node tt_node_matmul(tt_ctx* ctx, tt_node a, tt_node b);

/* a + b: b of a's shape, or b 1-D of a's last dimension, added to every row
 * (the bias of tinytorch 八.5). */
tt_node tt_node_add(tt_ctx* ctx, tt_node a, tt_node b);

/* a * b element by element, same shape (the scalar c = a * b of microcrad
 * for shape [1]). */
tt_node tt_node_mul(tt_ctx* ctx, tt_node a, tt_node b);

/* GELU, tanh form (tinytorch 三.4); its backward is the exact derivative of
 * that form. */
tt_node tt_node_gelu(tt_ctx* ctx, tt_node a);

/* Softmax over the last dimension, the row maximum subtracted first. */
tt_node tt_node_softmax(tt_ctx* ctx, tt_node a);

/* Cross entropy of probabilities p [R, C] at int32 labels y [R]:
 * -(1/R) sum_r ln p[r, y_r], a node of shape [1] (tinytorch 三.2
 * probs.CrossEntropy(y)).  A label outside [0, C) raises the context's bad
 * token flag (reported by tt_ctx_sync as TT_ERR_ARG) and counts as 0. */
tt_node tt_node_cross_entropy(tt_ctx* ctx, tt_node p, tt_node y);

/* Evaluate every non-leaf node that n depends on, and n, in creation order
 * (tinytorch 三.3 Forward). */
tt_status tt_node_forward(tt_ctx* ctx, tt_node n);

/* Zero the gradients of n and of every node it depends on (tinytorch 八.5
 * loss.ZeroGrad()). */
tt_status tt_node_zero_grad(tt_ctx* ctx, tt_node n);

/* Backpropagate from n: n's gradient is set to 1 (every element), the
 * gradients of the non-leaf nodes it depends on are cleared, and each of
 * them, in reverse creation order, adds its contribution (+=) into its
 * inputs' gradients; leaf gradients accumulate across calls until zeroed
 * (tinytorch 三.3; microcrad 反向传播).  When a cross entropy's input is a
 * softmax used by nothing else, the pair's gradient is formed directly as
 * (p - onehot(y)) / R (tinytorch 三.5). */
tt_status tt_node_backward(tt_ctx* ctx, tt_node n);

/* Copy count elements into n's values from src (host or device; f32 or
 * int32 per the node's type).  count must equal n's element count. */
tt_status tt_node_fill(tt_ctx* ctx, tt_node n, const void* src, size_t count);

/* Copy n's values (grad == 0) or gradient (grad != 0) to dst (host or
 * device), count = n's element count.  Synchronises the context's stream. */
tt_status tt_node_read(tt_ctx* ctx, tt_node n, int grad, void* dst, size_t count);

/* Shape and device buffers of n.  shape receives 4 ints (unused dims 1);
 * data/grad may be NULL; *grad is NULL for an int32 node. */
tt_status tt_node_info(tt_ctx* ctx, tt_node n, int* ndim, int* shape, void** data, float** grad);

/* SGD on the device: p[i] -= lr * grad[i] for every element of each of the
 * n_params f32 nodes (tinytorch 八.5). */
tt_status tt_node_sgd(tt_ctx* ctx, const tt_node* params, int n_params, float lr);

/* ---------------------------------------------------------------- recording
 * A fixed sequence of graph calls (a training step: forward, zero_grad,
 * backward, sgd) can be recorded once as a CUDA graph and replayed, so that
 * each later step costs one graph launch instead of one launch per kernel.
 * Between tt_capture_begin and tt_capture_end the calls of this header
 * record their kernels and memsets instead of running them; calls that must
 * wait for the device (tt_node_read, tt_node_fill from host memory,
 * tt_ctx_sync, tt_ctx_reset, the GPT-2 calls of tt.h) and calls that make
 * nodes return TT_ERR_STATE meanwhile.  A context keeps one recording: a new capture replaces it, and
 * tt_ctx_reset drops it (its nodes are gone). */

/* Start recording.  TT_ERR_STATE if a recording is already open. */
tt_status tt_capture_begin(tt_ctx* ctx);

/* Stop recording and keep what was recorded.  TT_ERR_STATE without an open
 * recording; TT_ERR_CUDA if a recorded call could not be captured (the
 * context is usable afterwards, with no recording). */
tt_status tt_capture_end(tt_ctx* ctx);

/* Run the recording `times` times on the context's stream, in order.
 * TT_ERR_STATE if there is no recording (or one is open), TT_ERR_ARG for
 * times < 0. */
tt_status tt_replay(tt_ctx* ctx, int times);

#ifdef __cplusplus
}
#endif
#endif /* TT_GRAPH_H */
