"""Device-memory plumbing around the C ABI: upload weights, own the model
handle, paged KV pools and workspaces.  Torch is used only to allocate and
copy; all compute goes through the binding."""
import numpy as np
import torch

from . import binding as B


def to_device_u16(arr: np.ndarray, device="cuda") -> torch.Tensor:
    """bf16 bit patterns (uint16) -> a bf16 tensor on `device`."""
    t = torch.from_numpy(np.ascontiguousarray(arr).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def make_config(shape, block=0, n_taps=0, conv_width=0, fc_norm=True, page_size=16):
    return B.DflashConfig(
        n_layers=shape.n_layers, hidden=shape.hidden, n_q_heads=shape.n_q_heads,
        n_kv_heads=shape.n_kv_heads, head_dim=shape.head_dim, mlp=shape.mlp,
        vocab=shape.vocab, block=block, n_taps=n_taps, conv_width=conv_width,
        qk_norm=1 if shape.qk_norm else 0, fc_norm=1 if fc_norm else 0,
        page_size=page_size, rms_eps=shape.rms_eps, rope_base=shape.rope_base,
        kv_terms=getattr(shape, "kv_terms", 1))


class DeviceModel:
    """Weights resident in HBM plus the library's model handle.

    ``weights`` / ``shared`` are dicts of uint16 (bf16-bit) NumPy arrays as
    produced by ``workload``; tensors already on the device are kept as is."""

    def __init__(self, shape, weights: dict, shared: dict, draft: bool, device="cuda"):
        self.shape = shape
        self.draft = draft
        self.t = {}
        for k, v in list(weights.items()) + list(shared.items()):
            self.t[k] = v if isinstance(v, torch.Tensor) else to_device_u16(v, device)
        w = B.DflashWeights()
        for f in B.WEIGHT_FIELDS:
            if f in self.t:
                setattr(w, f, self.t[f].data_ptr())
        if draft:
            cfg = make_config(shape, block=shape.block, n_taps=shape.n_taps,
                              conv_width=shape.conv_width, fc_norm=shape.fc_norm)
        else:
            cfg = make_config(shape)
        self.cfg = cfg
        self.weights_struct = w
        self.handle = B.dflash_model_create(cfg, w)

    def workspace(self, max_block_rows, max_ctx_rows, max_batch, max_ctx_len, device="cuda"):
        n = B.dflash_workspace_bytes(self.handle, max_block_rows, max_ctx_rows, max_batch,
                                     max_ctx_len)
        ws = torch.empty(n, dtype=torch.uint8, device=device)
        B.dflash_workspace_init(ws)
        return ws

    def close(self):
        if self.handle is not None and self.handle.value:
            B.dflash_model_destroy(self.handle)
        self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class PagedKV:
    """A paged KV pool [L][n_pages][2*kv_terms][hkv][page][d] and page table
    (planes K, V, then the low terms of K and V for a two-term cache).

    dtype "bf16": the pool holds bf16 values.  dtype "e4m3" (drafter context
    caches): the pool holds uint8 E4M3 codes [L][n_pages][2][hkv][page][d]
    and `scales` fp32 [L][n_pages][2][hkv][page], one per cached vector."""

    def __init__(self, shape, page_table: np.ndarray, n_pages: int, page_size=16,
                 device="cuda", zero=True, dtype="bf16"):
        L, hkv, d = shape.n_layers, shape.n_kv_heads, shape.head_dim
        planes = 2 * getattr(shape, "kv_terms", 1)
        alloc = torch.zeros if zero else torch.empty
        if dtype not in ("bf16", "e4m3"):
            raise ValueError(f"unknown cache dtype {dtype!r}")
        if dtype == "e4m3" and planes != 2:
            raise ValueError("E4M3 caches hold one term of K and V")
        self.dtype = dtype
        self.scales = None
        if dtype == "bf16":
            self.pool = alloc((L, n_pages, planes, hkv, page_size, d), dtype=torch.bfloat16,
                              device=device)
        else:
            self.pool = alloc((L, n_pages, 2, hkv, page_size, d), dtype=torch.uint8, device=device)
            self.scales = alloc((L, n_pages, 2, hkv, page_size), dtype=torch.float32,
                                device=device)
        self.table_np = np.ascontiguousarray(page_table, dtype=np.int32)
        self.table = torch.from_numpy(self.table_np).to(device)
        self.page_size = page_size
        self.n_pages = n_pages
        self.struct = B.DflashKV(pool=self.pool.data_ptr(), page_table=self.table.data_ptr(),
                                 n_pages=n_pages, max_pages=self.table_np.shape[1],
                                 n_rows=self.table_np.shape[0],
                                 dtype=0 if dtype == "bf16" else 1,
                                 scales=self.scales.data_ptr() if self.scales is not None else None)

    def quantized(self, model):
        """A new E4M3 cache with this bf16 cache's pages and table, every
        vector converted on the device (dflash_kv_quantize)."""
        if self.dtype != "bf16":
            raise ValueError("only a bf16 cache converts to E4M3")
        L, n_pages, _, hkv, page, d = self.pool.shape
        q = PagedKV.__new__(PagedKV)
        q.dtype = "e4m3"
        q.pool = torch.empty((L, n_pages, 2, hkv, page, d), dtype=torch.uint8,
                             device=self.pool.device)
        q.scales = torch.empty((L, n_pages, 2, hkv, page), dtype=torch.float32,
                               device=self.pool.device)
        q.table_np, q.table = self.table_np, self.table
        q.page_size, q.n_pages = self.page_size, self.n_pages
        q.struct = B.DflashKV(pool=q.pool.data_ptr(), page_table=q.table.data_ptr(),
                              n_pages=self.n_pages, max_pages=self.struct.max_pages,
                              n_rows=self.struct.n_rows, dtype=1, scales=q.scales.data_ptr())
        B.dflash_kv_quantize(model.handle, self.struct, q.struct)
        return q

    def read_codes(self, layer: int, req: int, n: int):
        """E4M3 cache: codes [n][2][hkv][d] (uint8) and scales [n][2][hkv] of
        one request's logical positions 0..n-1, on the host."""
        P = self.page_size
        idx = torch.arange(n, device=self.pool.device)
        pages = self.table[req].long()[idx // P]
        codes = self.pool[layer, pages, :, :, idx % P]
        scales = self.scales[layer, pages, :, :, idx % P]
        return codes.cpu().numpy(), scales.cpu().numpy()

    def fill_logical(self, layer: int, req: int, k_u16: np.ndarray, v_u16: np.ndarray):
        """Place already-projected context K/V ([len][hkv][d], bf16 bits) of
        one request at logical positions 0..len-1 (setup of a synthetic cache)."""
        n = k_u16.shape[0]
        P = self.page_size
        k = to_device_u16(k_u16, self.pool.device)
        v = to_device_u16(v_u16, self.pool.device)
        npg = (n + P - 1) // P
        pages = torch.from_numpy(self.table_np[req, :npg].astype(np.int64)).to(self.pool.device)
        pad = npg * P - n
        if pad:
            z = torch.zeros((pad,) + tuple(k.shape[1:]), dtype=k.dtype, device=k.device)
            k = torch.cat([k, z])
            v = torch.cat([v, z])
        # [npg][P][hkv][d] -> [npg][hkv][P][d]
        kk = k.view(npg, P, k.shape[1], k.shape[2]).transpose(1, 2)
        vv = v.view(npg, P, v.shape[1], v.shape[2]).transpose(1, 2)
        if pad:
            # keep slots past the end of the last page untouched
            full = npg - 1
            self.pool[layer, pages[:full], 0] = kk[:full]
            self.pool[layer, pages[:full], 1] = vv[:full]
            last = pages[full]
            keep = P - pad
            self.pool[layer, last, 0, :, :keep] = kk[full, :, :keep]
            self.pool[layer, last, 1, :, :keep] = vv[full, :, :keep]
        else:
            self.pool[layer, pages, 0] = kk
            self.pool[layer, pages, 1] = vv

    def read_logical(self, layer: int, req: int, n: int):
        """Context K/V of one request in logical order, as float32 tensors."""
        P = self.page_size
        idx = torch.arange(n, device=self.pool.device)
        pages = self.table[req].long()[idx // P]
        k = self.pool[layer, pages, 0, :, idx % P]
        v = self.pool[layer, pages, 1, :, idx % P]
        return k.float(), v.float()


def i32(x, device="cuda"):
    return torch.as_tensor(np.asarray(x, dtype=np.int32)).to(device)
