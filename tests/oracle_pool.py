"""Worker of the parity tests' pooled oracle: the wkv projection and the
gate of one token chunk, run by the single-threaded C oracle in a spawned
process.  Imports only numpy and the oracle, so workers start quickly."""
import numpy as np

import oracle


def oracle_chunk(args):
    (rows, w_path, ws, hidden, q, k, mask, eps, clamp, quantize_act, H, D) = args
    W_bits = np.ascontiguousarray(np.load(w_path, mmap_mode="r"))
    T = rows.shape[0]
    A = rows.reshape(T, -1)
    if ws is None:
        kv = oracle.wkv_bf16(A, W_bits)
    elif quantize_act:
        Aq, As = oracle.mx_quantize(A)
        kv = oracle.wkv_mxfp8_qact(Aq, As, W_bits, ws)
    else:
        kv = oracle.wkv_mxfp8(A, W_bits, ws)
    r = oracle.gate(hidden, kv, q, k, mask, eps, clamp)
    return dict(out_f64=r["out_f64"], out_bf16=r["out_bf16"], gate=r["gate"],
                value=np.ascontiguousarray(kv[:, H * D:]))
