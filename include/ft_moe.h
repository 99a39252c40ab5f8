/*
 * ft_moe.h -- C ABI of the routed, quantized expert-FFN MoE layer for GB300
 * (sm_103a).  One shared library, libft_moe.so, plain pointers and sizes.
 *
 * The layer, one call per step, all on one CUDA stream with no host sync:
 *   ft_moe_route          router logits, softmax, top-k
 *   ft_moe_resolve_slots  (layer, expert) -> cache slot or -1, q* split inside
 *   ft_moe_route_resolve  the two calls above with the top-k taken inside the
 *                         resolve kernel (one router grid, one resolve CTA)
 *   ft_moe_prefetch       speculative plan: the next layer's predicted misses
 *                         into eligible slots, one layer ahead of its resolve
 *   ft_moe_fetch          copy the chosen misses from the pool into the cache
 *   ft_moe_fetch_layer    copy a whole layer into a slot range (prefill buffer)
 *   ft_moe_cache_install  the state's bookkeeping for such a layer
 *   ft_moe_experts_fwd    quantized SwiGLU experts (decode: combine fused)
 *   ft_moe_permute        token permutation by expert (prefill)
 *   ft_moe_combine        top-k weighted sum of permuted expert rows (prefill)
 *   ft_moe_split_q16      the q* rule alone, batched (the resolve kernel runs
 *                         the same device function)
 *   ft_moe_decode_layer   route, resolve, fetch, experts and combine of one
 *                         decode layer call in one kernel
 *
 * Sources, by page title and section:
 *   "FreeToken 딥다이브" (fiv.co.kr) -- design pattern 1 (whole-layer double
 *     buffer for prefill), 2 (Q16 q* split inside the decode graph), 3 (-1
 *     sentinel and masking: every (token, expert) pair computed once),
 *     5 (slot LRU: int64 usage, global step, flat id layer*E+expert;
 *     expert_recency picks which misses are fetched).
 *   "FreeToken: 让消费级电脑跑起 284B MoE ..." (fengjutian.github.io) --
 *     sec. 2 (router on the GPU), sec. 4 (one slot = one (layer, expert);
 *     host pool is the source of truth), sec. 6 (q* = m*B_P/B_H; one kernel
 *     does dedup, residency, q, victims and id rewrite; exact merge),
 *     sec. 7 (banks with leading dimension layer*E+expert).
 *   "NVMe에서 전문가(experts)를 스트리밍하여 8GB GPU에서 133GB MoE 모델
 *     구동하기" (molayo1419.me) -- "Why this model" (three 2560x640 NVFP4
 *     matrices per expert), engine step 1 (one block per expert:
 *     gate|up|down|gate_scale|up_scale|down_scale), step 4 (single-token NVFP4
 *     SwiGLU expert kernel), step 5 (whole-prompt per-layer expert batching).
 *   "SSD 가중치층으로 35B MoE를 ..." (onedev.kr) -- "How it works":
 *     down(silu(gate(x)) * up(x)) over int4 weights, dedup/stack/gather.
 *
 * Conventions (all entry points):
 *   - Pointers named *_host are host memory; every other pointer is device
 *     accessible memory (cudaMalloc, or pinned host memory mapped into the
 *     device address space, e.g. the expert pool).  The caller owns all
 *     memory; no entry point allocates or frees device memory.
 *   - `stream` is a cudaStream_t passed as void*.  Calls only enqueue work;
 *     none synchronises the host, so a fixed-shape sequence of calls can be
 *     captured into a CUDA graph.
 *   - Return value: FT_OK, or an error found on the host before anything is
 *     enqueued (FT_ERR_INVALID: null pointer, bad size or range;
 *     FT_ERR_UNSUPPORTED: format/shape the kernels do not implement), or
 *     FT_ERR_CUDA when a launch fails.  ft_last_error() gives the message.
 *   - Errors that only the device can see (an expert id outside [0, E), a
 *     bounded wait that gave up) are recorded in the caller's int32
 *     `dev_status` word (first error wins, 0 = fine); the caller reads it
 *     after a synchronisation of its choosing.  dev_status may be NULL.
 *   - bf16 tensors are passed as uint16_t bit patterns.
 */
#ifndef FT_MOE_H
#define FT_MOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FT_API __attribute__((visibility("default")))
#else
#define FT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t ft_status;
enum {
  FT_OK = 0,
  FT_ERR_INVALID = 1,
  FT_ERR_UNSUPPORTED = 2,
  FT_ERR_CUDA = 3,
  FT_ERR_TIMEOUT = 4,   /* device: a bounded wait ran out */
  FT_ERR_BAD_ID = 5,    /* device: an expert id outside [0, E) */
  FT_ERR_RANGE = 6,     /* device: an intermediate left the f16 range (|h| > 2^20) */
  FT_ERR_REJECTED = 7   /* host: a cache rebuild that does not fit; nothing was changed */
};

/* Expert weight formats. */
enum {
  FT_INT4 = 0,   /* code q in 0..15 means (q - 8) * s; fp16 scale s per `group` K elements */
  FT_NVFP4 = 1   /* E2M1 code * E4M3 scale per 16 K elements * fp32 per-tensor scale */
};

enum { FT_DECODE = 0, FT_PREFILL = 1, FT_DECODE_HOST = 2 };
enum { FT_OUT_F32 = 0, FT_OUT_BF16 = 1 };
enum { FT_XP_BF16 = 0, FT_XP_F16 = 1 };  /* permuted-batch formats of ft_moe_permute */

/*
 * A bank: consecutive expert blocks (the pool indexed by flat id
 * fid = layer*E + expert, or the cache indexed by slot).  One block holds
 * gate [I,H] | up [I,H] | down [H,I] | gate_scale | up_scale | down_scale,
 * matrices row-major with K contiguous, two 4-bit codes per byte (low
 * nibble = even K).  Scales: int4 fp16 [rows, K/group]; NVFP4 E4M3 bytes
 * [rows, K/16].  Every block starts at base + index*stride; base and stride
 * must be multiples of 16 bytes; n_blocks is the number of blocks (kernels
 * skip, and record FT_ERR_BAD_ID for, any index outside it).  tensor_scale
 * (NVFP4 only) is a device
 * array [n_fids, 3] fp32 (gate, up, down) indexed by flat id, the same array
 * for pool and cache; NULL for int4.
 */
typedef struct {
  int32_t fmt;
  int32_t H;
  int32_t I;
  int32_t group;          /* int4: 32, 64 or 128; NVFP4: 16 */
  const void* base;
  uint64_t stride;
  int64_t n_blocks;
  const float* tensor_scale;
} ft_bank;

/*
 * The global slot cache state (device arrays, caller-owned), shared by all
 * layers.  slot_owner[S]: flat id held by the slot or -1.  map[L*E]: slot of
 * a flat id or -1.  usage[S]: last step the slot was used, -1 when empty.
 * recency[L*E]: last step the expert was routed.  step[1]: the global step,
 * advanced once per resolve call.
 */
typedef struct {
  int32_t L;
  int32_t E;
  int32_t S;
  int32_t* slot_owner;
  int32_t* map;
  int64_t* usage;
  int64_t* recency;
  int64_t* step;
} ft_cache_state;

/* Library and error queries. */
FT_API const char* ft_version(void);
FT_API const char* ft_status_string(ft_status s);
FT_API const char* ft_last_error(void);  /* message of the last failing call on this thread */

/*
 * Bytes of one expert block and the byte offsets of its six parts (off6 may
 * be NULL).  Returns 0 for an unsupported (fmt, H, I, group).
 */
FT_API uint64_t ft_block_bytes(int32_t fmt, int32_t H, int32_t I, int32_t group, uint64_t* off6_host);

/*
 * Copy the int32 status word to the host (synchronous: waits for the device
 * copy).  Use after the caller's own synchronisation point.
 */
FT_API ft_status ft_moe_get_status(const int32_t* dev_status, int32_t* out_host);

/*
 * ft_moe_route -- router on the GPU (FreeToken paper post, sec. 2).
 *   logits[t,e] = sum_h x[t,h] * w_router[e,h], fp32 accumulation;
 *   p = softmax over all E; topk_ids[t, 0..k-1] = experts by p descending,
 *   ties to the lower id; topk_w = p at those ids (divided by their sum when
 *   renorm != 0).
 * x [T,H] bf16 row-major; w_router [E,H] fp32 row-major; topk_ids [T,k]
 * int32; topk_w [T,k] fp32.  ws: device scratch of ft_moe_route_workspace(T,E,H)
 * bytes: an arrival counter in its first 256 bytes (T <= 16, where one
 * kernel computes the logits and its last CTA the top-k), then the logits,
 * then (T > 16, E a multiple of 128, H of 64: the logits on the tcgen05
 * tensor cores, summed over hidden slices of at most 1024) w_router split
 * exactly into three bf16 terms and the partial logits of every slice after
 * the first.
 * The counter sits at the same place for every T, so one workspace sized for
 * the largest T serves calls of any smaller T; ws must be zero-filled before
 * the first call that uses it, every call leaves the counter at zero, and
 * calls that may overlap on the GPU need separate workspaces.  Limits:
 * 1 <= k <= min(E, 32), E <= 4096, H % 8 == 0.  T == 0 is a no-op.
 */
FT_API size_t ft_moe_route_workspace(int32_t T, int32_t E, int32_t H);
FT_API ft_status ft_moe_route(const uint16_t* x, int32_t T, int32_t H, const float* w_router,
                       int32_t E, int32_t k, int32_t renorm, int32_t* topk_ids, float* topk_w,
                       void* ws, size_t ws_bytes, void* stream);

/*
 * ft_moe_split_q16 -- the bandwidth-matched q* rule in Q16 fixed point
 * (FreeToken deep-dive, design pattern 2; paper post, sec. 6).  For each m =
 * num_missing[i] and phi = frac_q16 = round(65536 * B_P / B_H):
 *   phi > 0: lo = (m*phi) >> 16; fetch lo or lo+1, whichever has the smaller
 *            max(f*(65536-phi), (m-f)*phi), ties to lo; capped at m.
 *   phi = 0: no cap, num_fetch = m.
 * num_missing, num_fetch: device int32 [n].  phi outside [0, 65536] or a
 * negative n is FT_ERR_INVALID.  Negative m gives 0.
 */
FT_API ft_status ft_moe_split_q16(const int32_t* num_missing, int32_t n, int32_t frac_q16,
                           int32_t* num_fetch, void* stream);

/*
 * ft_moe_resolve_slots -- one device kernel resolves a layer's top-k ids
 * against the global slot cache (FreeToken deep-dive, patterns 3 and 5;
 * paper post, sec. 6):
 *   U = distinct experts of ids (ascending); hits: map[layer*E+e] >= 0;
 *   m misses; num_fetch = min(q*(m, frac_q16), S - #hits); the fetched
 *   misses are the first num_fetch by (recency desc, id asc); the victims
 *   are the non-hit slots by (usage asc, slot asc), the i-th fetched expert
 *   taking the i-th victim; usage := step for hit and fetched slots;
 *   recency := step for all of U; step += 1; then
 *   slot_ids[t,j] = slot of ids[t,j] after the update, or -1 (host path).
 * topk_ids, slot_ids: [T,k] int32.  num_fetch: [1] int32.  fetch_fid,
 * fetch_slot: [max_list] int32, entries i < num_fetch hold (flat id, slot),
 * the rest -1; max_list >= min(T*k, S) is required.  An id outside [0, E)
 * records FT_ERR_BAD_ID in dev_status, leaves the state untouched and
 * writes slot_ids = -1, num_fetch = 0.  Limits: E <= 4096, T*k <= 4096.
 */
FT_API ft_status ft_moe_resolve_slots(const ft_cache_state* state_host, int32_t layer,
                               const int32_t* topk_ids, int32_t T, int32_t k,
                               int32_t frac_q16, int32_t* slot_ids, int32_t* num_fetch,
                               int32_t* fetch_fid, int32_t* fetch_slot, int32_t max_list,
                               int32_t* dev_status, void* stream);

/*
 * ft_moe_route_resolve -- ft_moe_route followed by ft_moe_resolve_slots
 * (FreeToken paper post, sec. 2: the router on the GPU feeding the hit /
 * miss split; sec. 6: one kernel dedups, checks residency, splits by q*,
 * picks victims and rewrites ids), with every output of those two calls:
 * topk_ids, topk_w, slot_ids, num_fetch, fetch_fid, fetch_slot and the
 * state update, bit for bit.  For T * k <= 32, E <= 512 and the state's
 * own E, the router grid writes only the logits and the resolve kernel takes
 * each token's softmax and top-k (one warp per token) before resolving,
 * which removes the router's arrival counter, its last CTA's top-k and the
 * reload of the ids from the chain.  Other shapes run the two calls in
 * order (larger calls resolve with the whole block, where the top-k in
 * front of it gained nothing).  Arguments as in the two calls: x [T,H] bf16, w_router [E,H] fp32
 * (both 16-byte aligned), route_ws of ft_moe_route_workspace(T,E,H) bytes
 * (zero-filled before its first use; this call leaves its counter as it
 * found it), the state, layer, frac_q16, slot_ids [T,k], num_fetch [1],
 * fetch_fid / fetch_slot [max_list], dev_status.  Invalid arguments of
 * either call are refused before anything is launched on the one-kernel
 * shapes.
 */
FT_API ft_status ft_moe_route_resolve(const uint16_t* x, int32_t T, int32_t H, const float* w_router,
                               int32_t E, int32_t k, int32_t renorm, int32_t* topk_ids,
                               float* topk_w, void* route_ws, size_t route_ws_bytes,
                               const ft_cache_state* state_host, int32_t layer, int32_t frac_q16,
                               int32_t* slot_ids, int32_t* num_fetch, int32_t* fetch_fid,
                               int32_t* fetch_slot, int32_t max_list, int32_t* dev_status,
                               void* stream);

/*
 * ft_moe_prefetch -- plan a speculative fetch of the next layer's experts
 * (NVMe-streaming post, "Where the time actually goes", speculative copies:
 * layer l+1's router run on layer l's MoE input picks most of layer l+1's
 * experts, so their copies can start one layer early, while layer l
 * computes).  pred_ids [T,k] int32 are the predicted ids of `layer` (from
 * ft_moe_route with that layer's router on the previous layer's input).  One
 * device kernel, the resolve's rules without the routing bookkeeping:
 *   U = distinct predicted experts; misses: map[layer*E+e] < 0, m of them;
 *   a slot may not be a victim if a predicted hit owns it, or if it is held
 *   (owner >= 0) with usage >= step-1 (the layer resolved last may still be
 *   reading it; usage == step marks an earlier prefetch not yet consumed);
 *   num_fetch = min(m, max_prefetch, eligible slots); the fetched misses are
 *   the first by (recency desc, id asc), the victims the eligible slots by
 *   (usage asc, slot asc), paired in order; victims' owners are evicted
 *   (map -1) and each victim takes its expert with usage = step.  Recency,
 *   hit usage and the step do not change.
 * Outputs have resolve's form (num_fetch [1]; fetch_fid / fetch_slot
 * [max_list], -1 after num_fetch; max_list >= min(T*k, S)), ready for
 * ft_moe_fetch on the same stream.  Ordering is the caller's: run it after
 * the resolve of the current layer and before the resolve of `layer`, and
 * let that layer's fetch and experts wait for the prefetch's copy.  An id
 * outside [0, E) records FT_ERR_BAD_ID, leaves the state untouched and
 * writes num_fetch = 0.  max_prefetch < 0 and the resolve's limits are
 * FT_ERR_INVALID.
 */
FT_API ft_status ft_moe_prefetch(const ft_cache_state* state_host, int32_t layer, const int32_t* pred_ids,
                                 int32_t T, int32_t k, int32_t max_prefetch, int32_t* num_fetch,
                                 int32_t* fetch_fid, int32_t* fetch_slot, int32_t max_list,
                                 int32_t* dev_status, void* stream);

/*
 * ft_moe_fetch -- copy each fetched expert block pool[fetch_fid[i]] ->
 * cache[fetch_slot[i]] for i < *num_fetch (read on the device, so the copy
 * count may come straight from resolve).  Pool and cache must have the same
 * format and shape; pool may be pinned host memory (the source of truth,
 * FreeToken paper post, sec. 4; deep-dive pattern 3 copy_missing).  A flat
 * id or slot outside its bank's n_blocks is skipped and records
 * FT_ERR_BAD_ID.
 */
FT_API ft_status ft_moe_fetch(const ft_bank* pool_host, const ft_bank* cache_host,
                       const int32_t* num_fetch, const int32_t* fetch_fid,
                       const int32_t* fetch_slot, int32_t max_list, int32_t* dev_status,
                       void* stream);

/*
 * ft_moe_fetch_layer -- copy every expert block of one layer, pool flat ids
 * layer*E .. layer*E+E-1, into cache slots slot0 .. slot0+E-1 with one
 * copy-engine transfer (no kernel: the SMs stay free for the experts).  It
 * is the load of prefill's whole-layer double buffer: layer l's experts in
 * slots (l%2)*E .., the next layer copied into the other half while this one
 * computes (FreeToken deep-dive, design pattern 1; paper post, sec. 5).
 * Pool and cache must have the same format and shape; the flat ids must be
 * inside the pool and the slots inside the cache (FT_ERR_INVALID otherwise,
 * checked on the host).  The cache state is not touched: pair it with
 * ft_moe_cache_install.
 */
FT_API ft_status ft_moe_fetch_layer(const ft_bank* pool_host, const ft_bank* cache_host, int32_t layer,
                                    int32_t E, int32_t slot0, void* stream);

/*
 * ft_moe_cache_install -- the slot cache's bookkeeping for a whole layer
 * placed in slots slot0 .. slot0+E-1 (the prefill double buffer above, which
 * then seeds decode).  With the end state of installing expert e = 0, 1, ..
 * in turn: a copy of flat id layer*E+e held in another slot outside the
 * range is dropped (owner -1, usage -1); the slot's previous owner is
 * evicted (map -1); slot slot0+e takes flat id layer*E+e with usage = the
 * current step.  Recency and the step are left alone (no routing happened).
 * Limits: E <= 4096, layer < L, slot0 + E <= S (FT_ERR_INVALID otherwise).
 * One small kernel on the stream; order it after the copy that fills the
 * slots when decode may run in between.
 */
FT_API ft_status ft_moe_cache_install(const ft_cache_state* state_host, int32_t layer, int32_t slot0,
                                      void* stream);

/*
 * ft_moe_cache_rebuild -- rebuild the slot cache at a new size (FreeToken
 * paper post, sec. 7 item 1: the GPU expert cache is re-partitioned at a
 * safe point for a new memory budget without reloading the host pool, which
 * stays the source of truth; deep-dive design pattern 7: everything is
 * validated before anything is destroyed, and a rebuild that does not fit is
 * refused).
 * Checks, on the host and before anything is enqueued: new_state has the
 * same L and E as old_state; new_cache the same format and shape as
 * old_cache and room for new_state->S blocks; new_state->S * new_cache->stride
 * plus 12 bytes per new slot (slot_owner, usage) fits in budget_bytes; and
 * the new bank and state arrays do not overlap the old ones.  Any failure
 * returns FT_ERR_REJECTED (FT_ERR_INVALID for a malformed call: NULL
 * pointers, negative sizes) and changes nothing.
 * Otherwise, on the stream: the resident experts of the old cache (slots
 * whose owner is >= 0) are ranked by usage, larger first, the lower slot
 * first among equals; the first min(residents, new S) move, in that order,
 * to new slots 0.. (block bytes copied old_cache -> new_cache, slot_owner and
 * usage carried over, map pointing at the new slots); every other new slot is
 * empty and every other flat id maps to -1; recency and step are copied.
 * The old state and bank are only read: the caller switches to the new ones
 * and frees the old after the stream has passed this call.  An old owner
 * outside [0, L*E) is skipped and records FT_ERR_BAD_ID.
 */
FT_API ft_status ft_moe_cache_rebuild(const ft_cache_state* old_state_host, const ft_bank* old_cache_host,
                                      const ft_cache_state* new_state_host, const ft_bank* new_cache_host,
                                      uint64_t budget_bytes, int32_t* dev_status, void* stream);

/*
 * ft_moe_experts_fwd -- quantized SwiGLU experts y = down(silu(gate.x) * up.x)
 * (SSD-tier Edge0 summary, "How it works"; NVMe post, step 4).
 * FT_DECODE: x [T,H] bf16; slot_ids, raw_ids, topk_w [T,k]; for each pair
 *   the expert block is cache[slot] when slot >= 0, else pool[layer*E + raw]
 *   when pool is non-NULL (the host-path pair, read in place), else the pair
 *   is skipped (masked: deep-dive pattern 3).  out [T,H] (FT_OUT_F32 or
 *   FT_OUT_BF16) = sum over computed pairs of topk_w * y, combine fused.
 *   h is kept in fp32.  Two pairs of one expert each read its rows (the
 *   repeat is served from L2).  Limits:
 *   T*k <= 256, T <= 16.  offsets unused (NULL).
 * FT_DECODE_HOST: as FT_DECODE but only the pairs with slot -1, read from
 *   pool (required); pairs with slot >= 0 are skipped.  With FT_DECODE on the
 *   cache alone (pool NULL) it splits one layer call into two disjoint
 *   partial sums that can run at the same time on two streams, the host path
 *   next to the fetch and the cache GEMV (deep-dive pattern 3: host work
 *   submitted first, the copy meanwhile, partial sums merged at the end;
 *   FreeToken paper post, sec. 6: the two branches add exactly);
 *   ft_moe_merge_partials adds them.
 * FT_PREFILL: x is the permuted batch Xp [T*k, H] in f16 as ft_moe_permute
 *   writes it with FT_XP_F16, x_scale [T*k] its per-row factors; offsets
 *   [E+1] its expert segments; slot_ids is a per-expert table [E] (the block
 *   of expert e is cache[slot_ids[e]]; every expert with rows must be
 *   resident, a -1 records FT_ERR_UNSUPPORTED); raw_ids and topk_w unused
 *   (NULL); out = Yp [T*k, H] bf16 (FT_OUT_BF16), the unweighted expert
 *   rows.  Runs on tcgen05 tensor cores with f16 operands: E2M1 x E4M3 is
 *   exact in f16, h is kept as f16(h / 16) (FT_ERR_RANGE if |h| > 2^20).
 *   NVFP4 only; H and I multiples of 256.
 * ws: device scratch of ft_moe_experts_workspace(...) bytes.
 */
FT_API size_t ft_moe_experts_workspace(int32_t mode, int32_t T, int32_t k, int32_t H, int32_t I,
                                int32_t E);
FT_API ft_status ft_moe_experts_fwd(const ft_bank* cache_host, const ft_bank* pool_host, int32_t layer,
                             int32_t E, const uint16_t* x, const float* x_scale, int32_t T,
                             const int32_t* slot_ids,
                             const int32_t* raw_ids, const float* topk_w, int32_t k,
                             int32_t mode, const int32_t* offsets, void* out, int32_t out_dtype,
                             void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * ft_moe_experts_decode_static -- ft_moe_experts_fwd in FT_DECODE mode with
 * no workspace argument: the scratch lives in a 1 MiB array of device memory
 * that the library owns (the source pages have no counterpart to this call).
 * It serves callers that cannot allocate device memory themselves -- code
 * running inside a stream capture, hosts whose GPU memory belongs to another
 * framework's pool, loops that cannot afford an allocation's synchronisation.
 * Same arguments and results as the decode mode above, minus ws.  Limits and
 * rules: ft_moe_experts_workspace(FT_DECODE, ...) = T*k*I*4 (rounded up to
 * 256) must not exceed 1 MiB (else FT_ERR_INVALID, nothing launched); every
 * GPU that loads the library keeps the array until exit;
 * calls that may overlap on the GPU share the array and race, so the caller
 * serialises them; the first call on a device looks the array up (with that
 * device current) and should happen before any stream capture.  The address
 * is kept for the life of the process, so the call must not be used on a
 * device after cudaDeviceReset (or any other reset of its primary context)
 * in the same process.
 */
FT_API ft_status ft_moe_experts_decode_static(const ft_bank* cache_host, const ft_bank* pool_host,
                                              int32_t layer, int32_t E, const uint16_t* x, int32_t T,
                                              const int32_t* slot_ids, const int32_t* raw_ids,
                                              const float* topk_w, int32_t k, void* out,
                                              int32_t out_dtype, int32_t* dev_status, void* stream);

/*
 * ft_moe_permute -- stable sort of the T*k (token, rank) pairs by expert
 * (expert asc, then token, then rank) and gather of the permuted batch
 * (NVMe post, step 5: the whole prompt through a layer's experts at once;
 * Edge0 "How it works": dedup, stack, gather).
 * topk_ids [T,k]; perm [T*k] (pair index t*k+j at each position); inv [T,k]
 * (position of each pair); offsets [E+1]; x [T,H] bf16 -> xp [T*k,H]
 * (NULL skips the gather).  xp_format FT_XP_BF16 copies the rows; FT_XP_F16
 * writes f16(x * 2^-s) with s >= 0 the smallest power of two keeping the
 * row below 2^15, and xp_scale[pos] = 2^s (exact; the grouped experts kernel
 * multiplies its results by it).  ws: ft_moe_permute_workspace(T,k,E) bytes.
 * An id outside [0, E) records FT_ERR_BAD_ID.  Limits: E <= 4096.
 */
/*
 * ft_moe_decode_layer -- one decode layer call, the whole hot path in one
 * kernel launch: ft_moe_route, ft_moe_resolve_slots (q* split inside),
 * ft_moe_fetch and ft_moe_experts_fwd(FT_DECODE) with the pool as host path,
 * in that order and with the same results (FreeToken paper post, secs. 2 and
 * 6: router on the GPU, one kernel for dedup, residency, q, victims and the
 * id rewrite, no host crossing in the layer; FreeToken deep-dive, design
 * patterns 2, 3 and 5; SSD-tier 35B post, "How it works"; NVMe-streaming
 * post, step 4).
 * x [T,H] bf16; w_router [E,H] fp32 (E = state->E, H = the bank's); outputs
 * as the separate calls write them: topk_ids/topk_w [T,k], slot_ids [T,k],
 * *num_fetch, fetch_fid/fetch_slot [max_list], out [T,H] (out_dtype).  The
 * pool (the source of truth) is required: fetched experts are copied from
 * it and pairs left on slot -1 read it in place.  ws: device scratch of
 * ft_moe_decode_layer_workspace(T,k,H,I,E) bytes, 256-byte aligned: a
 * counter and a generation word in its first 256 bytes, then the logits and
 * h.  ws must be zero-filled before the first call that uses it; every call
 * leaves the counter at zero, so one workspace serves every later call of
 * any shape it is large enough for; calls that may overlap on the GPU need
 * separate workspaces.
 * The grid is one CTA per SM, launched cooperatively (its CTAs wait for one
 * another through the workspace, each wait bounded by ft_set_wait_limit_ns);
 * a wait that gives up records FT_ERR_TIMEOUT in dev_status, the kernel
 * returns, and later calls that see that status do nothing: the caller then
 * zero-fills ws and the status word before calling again.
 * Limits: 1 <= T <= 8, T*k <= 128, k <= min(E, 32), E <= 512 and
 * E <= 4 x the SM count, H and I <= 4096, bank blocks 16-byte aligned, and
 * the call's shared-memory plan must fit one SM (FT_ERR_INVALID otherwise,
 * nothing launched; the separate calls serve those shapes).
 */
FT_API size_t ft_moe_decode_layer_workspace(int32_t T, int32_t k, int32_t H, int32_t I, int32_t E);
FT_API ft_status ft_moe_decode_layer(const uint16_t* x, int32_t T, const float* w_router, int32_t k,
                              int32_t renorm, const ft_cache_state* state_host, int32_t layer,
                              int32_t frac_q16, const ft_bank* cache_host, const ft_bank* pool_host,
                              int32_t* topk_ids, float* topk_w, int32_t* slot_ids, int32_t* num_fetch,
                              int32_t* fetch_fid, int32_t* fetch_slot, int32_t max_list, void* out,
                              int32_t out_dtype, void* ws, size_t ws_bytes, int32_t* dev_status,
                              void* stream);

/*
 * ft_set_wait_limit_ns -- the limit of every bounded wait inside the kernels
 * launched after this call (the decode layer's hand-offs and copy waits),
 * in nanoseconds of the GPU's global timer; 0 restores the default of 2 s.
 * Process-wide; not tied to a device or stream.  Always FT_OK.
 */
FT_API ft_status ft_set_wait_limit_ns(uint64_t ns);

FT_API size_t ft_moe_permute_workspace(int32_t T, int32_t k, int32_t E);
FT_API ft_status ft_moe_permute(const int32_t* topk_ids, int32_t T, int32_t k, int32_t E,
                         const uint16_t* x, int32_t H, int32_t* perm, int32_t* inv,
                         int32_t* offsets, uint16_t* xp, int32_t xp_format, float* xp_scale,
                         void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/*
 * ft_moe_merge_partials -- out[i] = a[i] + b[i] for i < n (fp32 inputs;
 * out fp32 or bf16 by out_dtype): the final merge of a decode layer call
 * split into its cache and host-path partial sums (FT_DECODE on the cache,
 * FT_DECODE_HOST on the pool).  out may alias a or b.
 */
FT_API ft_status ft_moe_merge_partials(const float* a, const float* b, int64_t n, void* out,
                                       int32_t out_dtype, void* stream);

/*
 * ft_moe_combine -- out[t] = sum_j topk_w[t,j] * yp[inv[t,j]] in j order,
 * fp32 accumulation, plus host_partial[t] when non-NULL (the host path's
 * partial sum: FreeToken paper post, sec. 6, exact merge), rounded to bf16.
 * yp [T*k,H] bf16; inv, topk_w [T,k]; host_partial [T,H] fp32; out [T,H] bf16.
 */
FT_API ft_status ft_moe_combine(const uint16_t* yp, const int32_t* inv, const float* topk_w,
                         int32_t T, int32_t k, int32_t H, const float* host_partial,
                         uint16_t* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FT_MOE_H */
