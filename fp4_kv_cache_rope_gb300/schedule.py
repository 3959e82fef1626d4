"""The CSA2 layer schedule of one decode token through the whole model.

Host-side orchestration only: which C-ABI call each layer makes, on which
cache, with which selection.  Every step of the arithmetic runs in the kernels
behind ``include/csa2.h``.

The schedule the pages give ("DeepSeek-V4.1-Flash: Pushing the Limits of KV
Cache Compression" knowledge note, section "CSA2: share cache, refresh
selection only when needed" and its symbol table; "The 890-Byte Token",
section "CSA2 cross-layer KV and index reuse"):

* 40 layers: a 20-layer causal encoder, then a 20-layer decoder.
* Encoder: three CSA2 groups, each a Full layer (2, 8, 14) followed by five
  Reuse layers; each group owns a cache of m = 2 entries (two source
  positions per entry).
* Decoder: one cache of m = 1 entries written by the Full layer 20 (followed
  by three Reuse layers), then four groups of a Reindex layer (24, 28, 32, 36)
  over layer 20's pool followed by three Reuse layers.
* Layers 0 and 1 use no global branch (4 Full + 4 Reindex + 30 Reuse = the 38
  CSA2 layers the pages count).

Every CSA2 layer computes its own query and SWA window and attends; Reuse
layers take the most recent selection of their group.  The layers of a group
share one cache and one selection, so their attentions go to the GPU together:
one ``csa2_attn_decode_layers`` launch serves up to ``floor(SMs / B)`` of them
(at most ``MAX_ATTN_LAYERS``), which fills the SMs with whole sequences
instead of splitting each sequence's keys over several CTAs and merging.
"""
from __future__ import annotations

from dataclasses import dataclass

FULL, REINDEX, REUSE = 0, 1, 2
N_LAYERS = 40
ENCODER_FULL = (2, 8, 14)
ENCODER_GROUP = 6          # Full + 5 Reuse
DECODER_FULL = 20
DECODER_REINDEX = (24, 28, 32, 36)
DECODER_GROUP = 4          # Full or Reindex + 3 Reuse


@dataclass(frozen=True)
class LayerPlan:
    layer: int
    mode: int          # FULL, REINDEX or REUSE
    cache: int         # 0..2: encoder group caches (m = 2); 3: the decoder cache (m = 1)
    selection: int     # the index-producing layer whose top-k this layer attends over


def layer_plan() -> list:
    """The 38 CSA2 layers of the model, in order."""
    plan = []
    for layer in range(2, N_LAYERS):
        if layer < DECODER_FULL:
            g = (layer - ENCODER_FULL[0]) // ENCODER_GROUP
            head = ENCODER_FULL[g]
            plan.append(LayerPlan(layer, FULL if layer == head else REUSE, g, head))
        else:
            head = DECODER_FULL + (layer - DECODER_FULL) // DECODER_GROUP * DECODER_GROUP
            if layer == DECODER_FULL:
                mode = FULL
            elif layer in DECODER_REINDEX:
                mode = REINDEX
            else:
                mode = REUSE
            plan.append(LayerPlan(layer, mode, 3, head))
    return plan


def attention_chunks(plan, per_launch: int) -> list:
    """The plan's layers cut into attention launches: consecutive layers with
    the same cache and selection, at most per_launch of them per launch."""
    chunks = []
    for p in plan:
        c = chunks[-1] if chunks else None
        if (c and len(c) < per_launch and c[0].cache == p.cache
                and c[0].selection == p.selection):
            c.append(p)
        else:
            chunks.append([p])
    return chunks


class DecodeSchedule:
    """Runs the 38 CSA2 layers of one decode token for a batch of sequences.

    caches:     four Cache objects: the three encoder caches (m = 2 entries)
                and the decoder cache (m = 1).
    workspaces: one workspace per cache (calls on a cache share its workspace;
                all calls go to one stream, in order).
    topk, window, heads, idx_heads: the layer shapes (shared by all layers).
    """

    def __init__(self, caches, workspaces, heads, idx_heads, topk, window, layers_per_launch=None):
        import torch
        from . import MAX_ATTN_LAYERS, POOL_BLOCKS
        assert len(caches) == 4 and len(workspaces) == 4
        self.caches, self.ws = caches, workspaces
        self.heads, self.idx_heads, self.topk, self.window = heads, idx_heads, topk, window
        self.plan = layer_plan()
        B = caches[3].batch
        dev = caches[3].codes.device
        if layers_per_launch is None:
            sms = torch.cuda.get_device_properties(dev).multi_processor_count
            layers_per_launch = sms // B
        self.layers_per_launch = max(1, min(MAX_ATTN_LAYERS, int(layers_per_launch)))
        self.chunks = attention_chunks(self.plan, self.layers_per_launch)
        heads_ = {p.selection for p in self.plan}
        self.idx = {h: torch.zeros((B, topk), dtype=torch.int32, device=dev) for h in heads_}
        self.cnt = {h: torch.zeros((B,), dtype=torch.int32, device=dev) for h in heads_}
        self.pool = torch.zeros((B, 1, POOL_BLOCKS), dtype=torch.int32, device=dev)
        self.pool_cnt = torch.zeros((B, 1), dtype=torch.int32, device=dev)

    def append(self, dec_kv, dec_idx, enc=None):
        """Append the token: one decoder entry, and -- when the token completes
        a pair -- one entry to each encoder cache.  enc: three (kv, z, idx)
        triples of [B, 2, D], [B, 2, D], [B, 1, di] tensors, or None."""
        from . import quant_append, quant_append_pairs
        quant_append(self.caches[3], dec_kv, dec_idx, 1, self.ws[3])
        if enc is not None:
            for g in range(3):
                kv, z, ik = enc[g]
                quant_append_pairs(self.caches[g], kv, z, ik, 1, self.ws[g])

    def layers(self, inputs, out, on_layer=None):
        """Index and attend every CSA2 layer.

        inputs[layer]: dict with q (bf16 [B, H, D] as int16), swa (E4M3 [B, W, D])
                       and, for Full / Reindex layers, q_idx (E4M3 [B, 1, Hi, di])
                       and w (fp32 [B, 1, Hi]).
        out[layer]:    fp32 [B, H, D], written.
        on_layer(plan_entry, phase, before): optional hook called before and
                       after each call, e.g. for events.  phase "index" names
                       the indexing layer; phase "attention" names the first
                       layer of the launch (``self.chunks``).
        """
        from . import attn_decode, attn_decode_layers, index_full, index_reindex
        B, k = self.caches[3].batch, self.topk
        for chunk in self.chunks:
            p = chunk[0]
            c, ws = self.caches[p.cache], self.ws[p.cache]
            if p.mode != REUSE:
                inp = inputs[p.layer]
                h = p.selection
                sel = self.idx[h].view(B, 1, k)
                cnt = self.cnt[h].view(B, 1)
                if on_layer:
                    on_layer(p, "index", True)
                if p.mode == FULL:
                    dec = p.cache == 3       # the decoder Full layer keeps the pool
                    index_full(c, inp["q_idx"], inp["w"], self.idx_heads, 1, None, None, B, k,
                               sel, cnt, self.pool if dec else None,
                               self.pool_cnt if dec else None, ws)
                else:
                    index_reindex(c, inp["q_idx"], inp["w"], self.idx_heads, 1, None, self.pool,
                                  self.pool_cnt, None, B, k, sel, cnt, ws)
                if on_layer:
                    on_layer(p, "index", False)
            if on_layer:
                on_layer(p, "attention", True)
            if len(chunk) == 1:
                inp = inputs[p.layer]
                attn_decode(c, inp["q"], self.heads, self.idx[p.selection], self.cnt[p.selection],
                            k, inp["swa"], None, self.window, 0.0, out[p.layer], ws)
            else:
                attn_decode_layers(c, [inputs[x.layer]["q"] for x in chunk], self.heads,
                                   self.idx[p.selection], self.cnt[p.selection], k,
                                   [inputs[x.layer]["swa"] for x in chunk], None, self.window,
                                   0.0, [out[x.layer] for x in chunk], ws)
            if on_layer:
                on_layer(p, "attention", False)

    def launches(self, pair_appended):
        """Kernel launches of one token (append clusters, 2 per index call, 1
        per attention launch)."""
        n = 1 + (3 if pair_appended else 0)
        n += sum(2 for p in self.plan if p.mode != REUSE)
        n += len(self.chunks)
        return n
