"""Model wrappers: upload seeded weights to the GPU and create a lat context.

PyTorch is used only to hold device memory and streams; all arithmetic of the
path runs in liblat.so.
"""
import numpy as np
import torch

from . import lat


def _dev_bf16(bits, device) -> torch.Tensor:
    """Upload bf16 bit patterns (uint16 array) as a torch bfloat16 tensor; a
    bfloat16 torch tensor is taken as it is (moved to `device` if needed)."""
    if isinstance(bits, torch.Tensor):
        assert bits.dtype == torch.bfloat16, "weights must be bfloat16"
        return bits.to(device).contiguous()
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def desc_from_config(cfg: dict, kind: int, max_batch: int = 1, n_streams: int = 1) -> lat.ModelDesc:
    d = lat.ModelDesc()
    d.kind = kind
    d.D = cfg["D"]
    if cfg["kind"] == "dit":
        d.Hq = d.Hkv = cfg["H"]
    else:
        d.Hq, d.Hkv = cfg["Hq"], cfg["Hkv"]
    d.dh, d.F, d.L = cfg["dh"], cfg["F"], cfg["L"]
    d.S = cfg.get("S", 0)
    d.T_prefix = cfg.get("T_prefix", 0) if cfg["kind"] != "dit" else 0
    d.T_q = cfg["T_chunk"] if cfg["kind"] == "dit" else cfg["T_q"]
    d.act_dim = cfg.get("act_dim", 0)
    d.n_hist = cfg.get("n_hist", 0)
    d.t_dim = cfg.get("t_dim", 0)
    d.patch_dim = cfg.get("patch_dim", 0)
    d.max_batch = max_batch
    d.n_streams = n_streams
    d.rope_base = cfg["rope_base"]
    d.eps = cfg["eps"]
    d.prefix_lm = int(cfg.get("prefix_lm", 0))
    d.grid_h = cfg.get("grid_h", 0)
    d.grid_w = cfg.get("grid_w", 0)
    d.text_len = cfg.get("text_len", 0)
    d.page_tokens = cfg.get("page_tokens", 0)
    return d


class Pi0ActionExpert:
    """The pi0 action expert behind lat_denoise_chunk / lat_block_forward."""

    def __init__(self, cfg: dict, weight_bits: dict, device="cuda"):
        self.cfg = cfg
        self.device = torch.device(device)
        keep = []

        def up(x):
            t = _dev_bf16(x, self.device)
            keep.append(t)
            return lat.ptr(t)

        L = cfg["L"]
        blocks = (lat.BlockWeights * L)()
        for l, b in enumerate(weight_bits["blocks"]):
            for k in ("g_attn", "wq", "wk", "wv", "wo", "g_ffn", "wg", "wu", "wd"):
                setattr(blocks[l], k, up(b[k]))
        w = lat.Weights()
        w.blocks = blocks
        for k in ("w_in", "b_in", "w1", "b1", "w2", "b2", "w_state", "b_state", "g_final", "w_out", "b_out"):
            setattr(w, k, up(weight_bits[k]))
        self._blocks = blocks
        self.ctx = lat.Context(desc_from_config(cfg, lat.LAT_PI0_ACTION_EXPERT), w)
        torch.cuda.synchronize()
        del keep  # the library folded its own copies

    def kv_from_bits(self, kv_bits: np.ndarray) -> torch.Tensor:
        return _dev_bf16(kv_bits, self.device)

    def denoise(self, kv: torch.Tensor, state: torch.Tensor, x: torch.Tensor, stream=None):
        self.ctx.denoise_chunk(kv, state, x, stream)

    def block(self, layer: int, x: torch.Tensor, kv_layer: torch.Tensor, stream=None):
        self.ctx.block_forward(layer, x, kv_layer, None, stream)


def bits_of(t: torch.Tensor) -> np.ndarray:
    """bf16 torch tensor -> uint16 bit patterns (host)."""
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


class _Uploader:
    def __init__(self, device):
        self.device = device
        self.keep = []

    def __call__(self, bits):
        t = _dev_bf16(bits, self.device)
        self.keep.append(t)
        return lat.ptr(t)


class Pi0Prefix:
    """The prefix model behind lat_prefill_kv (per-layer K/V of the vision tokens)."""

    def __init__(self, cfg: dict, weight_bits: dict, max_batch: int = 1, device="cuda"):
        self.cfg = cfg
        self.device = torch.device(device)
        up = _Uploader(self.device)
        blocks = (lat.BlockWeights * cfg["L"])()
        for l, b in enumerate(weight_bits["blocks"]):
            for k in ("g_attn", "wq", "wk", "wv", "wo", "g_ffn", "wg", "wu", "wd"):
                setattr(blocks[l], k, up(b[k]))
        w = lat.Weights()
        w.blocks = blocks
        w.w_patch = up(weight_bits["w_patch"])
        w.b_patch = up(weight_bits["b_patch"])
        self._blocks = blocks
        self.ctx = lat.Context(desc_from_config(cfg, lat.LAT_PI0_PREFIX, max_batch=max_batch), w)
        torch.cuda.synchronize()

    def new_kv(self, B):
        c = self.cfg
        return torch.zeros((c["L"], B, 2, c["T_prefix"] + c["T_q"], c["Hkv"] * c["dh"]),
                           dtype=torch.bfloat16, device=self.device)

    def prefill(self, patch_emb: torch.Tensor, kv: torch.Tensor, stream=None):
        self.ctx.prefill_kv(patch_emb, patch_emb.shape[0], kv, stream)


class DitStage:
    """One DiT stage (L blocks) behind lat_block_forward."""

    def __init__(self, cfg: dict, weight_bits: dict, max_batch: int = 4, n_streams: int = 1, device="cuda"):
        self.cfg = cfg
        self.device = torch.device(device)
        up = _Uploader(self.device)
        L = len(weight_bits["blocks"])
        blocks = (lat.BlockWeights * L)()
        for l, b in enumerate(weight_bits["blocks"]):
            for k in ("wq", "wk", "wv", "wo", "w1", "w2"):
                setattr(blocks[l], k, up(b[k]))
            if cfg.get("text_len", 0):
                for k, f in (("g_c", "g_cross"), ("b_c", "b_cross"), ("cq", "cq"), ("ck", "ck"), ("cv", "cv"),
                             ("co", "co")):
                    setattr(blocks[l], f, up(b[k]))
        w = lat.Weights()
        w.blocks = blocks
        for k in ("wt1", "bt1", "wt2", "bt2", "wmod", "bmod"):
            setattr(w, k, up(weight_bits[k]))
        # latent in/out projections of the stage (interleaved schedule), when given
        latent_io = "w_in" in weight_bits and cfg.get("lat_dim", 0) > 0
        if latent_io:
            for k in ("w_in", "b_in", "w_out", "b_out"):
                setattr(w, k, up(weight_bits[k]))
        self._blocks = blocks
        cfg = dict(cfg, L=L)
        self.cfg = cfg
        desc = desc_from_config(cfg, lat.LAT_DIT, max_batch=max_batch, n_streams=n_streams)
        desc.act_dim = cfg["lat_dim"] if latent_io else 0
        self.ctx = lat.Context(desc, w)
        torch.cuda.synchronize()

    def interval(self, ring: torch.Tensor, lat_z: torch.Tensor, chunks, stream=None):
        """One interval of the interleaved schedule on latents lat_z [n][T][lat_dim] (in place)."""
        self.ctx.dit_interval(ring, lat_z, chunks, stream=stream)

    def push(self, ring: torch.Tensor, stream_id: int, noise=None, done=None, stream=None) -> int:
        return self.ctx.dit_pipeline_push(ring, stream_id, noise, done, stream=stream)

    def block(self, layer, x: torch.Tensor, chunks, ring: torch.Tensor, stream=None):
        self.ctx.block_forward(layer, x, ring, chunks=chunks, stream=stream)

    def set_text(self, stream_id: int, text_bits, stream=None):
        """The text context of one stream: bf16 bits [text_len][D] (host numpy) or a
        bf16 device tensor."""
        t = _dev_bf16(text_bits, self.device)
        self.ctx.dit_set_text(stream_id, t, stream=stream)
        self._text_keep = getattr(self, "_text_keep", {})
        self._text_keep[stream_id] = t   # read by the enqueued work

    def bind_pages(self, table):
        """The page table (int32 [n_streams][L][S][pages], host numpy or device tensor)."""
        t = table if isinstance(table, torch.Tensor) else torch.from_numpy(table)
        t = t.to(self.device, dtype=torch.int32).contiguous()
        self._pages = t
        self.ctx.dit_bind_pages(t)
