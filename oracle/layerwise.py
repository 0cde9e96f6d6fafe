"""CPU oracle of layerwise prefill offload.  TEST INFRASTRUCTURE ONLY: the tests,
the smoke check and the benchmark's CPU legs use it; the library never does.

Source: "Layerwise and Sparse KV Cache Offloading Design", section 3
"Layerwise Prefill Offload" ("Buffer planning", "Execution pipeline", "Reuse
invariant"), and the FlashOffloading explainer's prefill paragraph (four trays,
tray B0 bound to the first layer, onload_layer_map lookahead).

Readings (choices of this project where the pages leave a step open):
 R14 plan      : N cache-bearing layers, a set of independent layers with a
                 dedicated buffer each (default: layer 0, the explainer's tray B0),
                 B shared buffers.  physical buffers = I + min(B, R), R = N - I.
                 Independent layers take buffers 0..I-1 in layer order; the R
                 reusable layers, in layer order, take shared buffer
                 I + (k mod min(B, R)) for the k-th of them (round robin).  One
                 uniform cache layout, so every reusable layer is compatible.
 R15 pass      : one prefill forward pass over a chunk of c new tokens with a
                 cached prefix of L tokens.  For each layer in order: the layer's
                 buffer holds rows 0..L-1 of its main-KV history (loaded from the
                 host pool unless the buffer already holds them: an independent
                 layer keeps its buffer across passes); the layer's compute reads
                 them and writes the chunk's rows at L..L+c-1; the save copies rows
                 L..L+c-1 back to the host pool.  After the pass L += c.  A buffer
                 is reused only after the save of its previous layer has finished
                 (the reuse invariant), and the load of a layer may start up to
                 `lookahead` layers ahead of its compute.
 R16 stand-in  : the tests' stand-in for the layer's attention and KV update reads the
                 whole cached prefix of the layer and reports its digest, the exact
                 sum of its bf16 bit patterns taken as unsigned 16-bit integers, so
                 that a load that brought the wrong rows, or a buffer overwritten
                 before the compute read it, changes the digest.
"""
import numpy as np


def plan(n_layers, independent=(0,), n_shared=3):
    """R14: (n_phys, phys_of_layer) for a uniform layout."""
    if n_layers < 1 or n_shared < 0:
        raise ValueError("n_layers >= 1 and n_shared >= 0")
    ind = sorted(set(int(l) for l in independent))
    if any(l < 0 or l >= n_layers for l in ind):
        raise ValueError("independent layer out of range")
    reusable = [l for l in range(n_layers) if l not in ind]
    r = len(reusable)
    shared = min(n_shared, r)
    if r > 0 and shared == 0:
        raise ValueError("reusable layers need at least one shared buffer")
    phys = [-1] * n_layers
    for k, l in enumerate(ind):
        phys[l] = k
    for k, l in enumerate(reusable):
        phys[l] = len(ind) + (k % shared)
    return len(ind) + shared, phys


def footprint_ratio(n_layers, n_phys):
    """Main-KV device footprint of the plan relative to every layer resident."""
    return n_phys / n_layers


def digest(rows):
    """R16: exact sum of the bf16 bit patterns (unsigned 16-bit) of rows."""
    return int(np.asarray(rows, dtype=np.uint16).astype(np.int64).sum())


class LayerwiseOracle:
    """R15: the host pool of one request across prefill passes."""

    def __init__(self, n_layers, max_tokens, row_elems=576):
        self.n_layers, self.max_tokens, self.row_elems = n_layers, max_tokens, row_elems
        self.host = np.zeros((n_layers, max_tokens, row_elems), dtype=np.uint16)
        self.length = 0

    def fill_prefix(self, rows):
        """rows: [n_layers][L][row_elems] uint16, the cached prefix before the first pass."""
        rows = np.asarray(rows, dtype=np.uint16)
        L = rows.shape[1]
        if L > self.max_tokens:
            raise ValueError("prefix longer than max_tokens")
        self.host[:, :L] = rows
        self.length = L

    def forward(self, chunk):
        """One pass: chunk [n_layers][c][row_elems] uint16.  Returns the per-layer digests
        the stand-in compute reads (of rows 0..L-1 before the chunk is written)."""
        chunk = np.asarray(chunk, dtype=np.uint16)
        c = chunk.shape[1]
        if self.length + c > self.max_tokens:
            raise ValueError("pass past max_tokens")
        digests = []
        for l in range(self.n_layers):
            digests.append(digest(self.host[l, :self.length]))
            self.host[l, self.length:self.length + c] = chunk[l]
        self.length += c
        return digests
