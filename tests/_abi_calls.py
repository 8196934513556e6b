"""Argument checks of the C ABI that need non-null pointers, run in a child process with no
visible CUDA device (CUDA_VISIBLE_DEVICES=""), so that no call can reach a launch whatever
the order of the checks.  The pointers are host buffers, never device addresses.  Prints one
JSON object of status codes; tests/test_abi.py runs it."""
import ctypes
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from gated_linear_sliding_gb300 import lizard as lz  # noqa: E402


def dims(**kw):
    base = dict(B=1, L=128, Hq=32, Hkv=8, d=128, D=128, w=64, M=4, dtype=lz.LIZARD_BF16,
                decay=lz.LIZARD_DECAY_DELAYED)
    base.update(kw)
    return lz.make_dims(base["B"], base["L"], base["Hq"], base["Hkv"], base["d"], base["D"],
                        base["w"], base["M"], base["dtype"], decay=base["decay"])


def main():
    assert os.environ.get("CUDA_VISIBLE_DEVICES") == "", "must run without a visible device"
    lib = lz.load()
    buf = ctypes.create_string_buffer(4096 + 64)
    base = (ctypes.addressof(buf) + 63) & ~63
    ok = ctypes.c_void_p(base)           # 16-byte aligned host address
    mis = ctypes.c_void_p(base + 4)      # misaligned host address
    out = {}
    d = dims()
    args = [ok] * 7 + [None] * 5 + [ok]
    out["fwd_null_q"] = lib.lizard_attn_fwd(ctypes.byref(d), None, *args[1:], 1 << 30, None)
    a2 = list(args)
    a2[2] = mis
    out["fwd_misaligned_v"] = lib.lizard_attn_fwd(ctypes.byref(d), *a2, 1 << 30, None)
    a3 = list(args)
    a3[8] = ok  # S_out without z_out
    out["fwd_S_without_z"] = lib.lizard_attn_fwd(ctypes.byref(d), *a3, 1 << 30, None)
    a4 = list(args)
    a4[12] = mis
    out["fwd_misaligned_ws"] = lib.lizard_attn_fwd(ctypes.byref(d), *a4, 1 << 30, None)
    d96 = dims(d=96, D=96)
    out["fwd_unsupported"] = lib.lizard_attn_fwd(ctypes.byref(d96), *args, 1 << 30, None)
    need = lz.lizard_attn_fwd_workspace(d)
    out["fwd_small_ws"] = lib.lizard_attn_fwd(ctypes.byref(d), *args, need - 16, None)
    out["noalloc_misaligned"] = lib.lizard_attn_fwd_noalloc(ctypes.byref(d), *a2[:12], None)
    nul = [ok] * 13  # q .. vcache, gcache
    out["dec_w300"] = lib.lizard_decode_step(ctypes.byref(dims(w=300)), 0, *nul, 256, None)
    out["dec_G16"] = lib.lizard_decode_step(ctypes.byref(dims(Hq=32, Hkv=2)), 0, *nul, 256, None)
    out["dec_neg_pos"] = lib.lizard_decode_step(ctypes.byref(dims()), -1, *nul, 256, None)
    out["dec_misaligned"] = lib.lizard_decode_step(ctypes.byref(dims()), 0, mis, *nul[1:], 256,
                                                   None)
    # decay readings: an unknown one, and a masked/lagged decode without its gate ring
    out["fwd_bad_decay"] = lib.lizard_attn_fwd(ctypes.byref(dims(decay=3)), *args, 1 << 30, None)
    for name, code in (("masked", lz.LIZARD_DECAY_MASKED), ("lagged", lz.LIZARD_DECAY_LAGGED)):
        # nul[:11] = q .. vcache, then gcache, workspace, its size, the stream
        out[f"dec_{name}_no_gcache"] = lib.lizard_decode_step(
            ctypes.byref(dims(decay=code)), 0, *nul[:11], None, ok, 1 << 20, None)
        out[f"dec_{name}_mis_gcache"] = lib.lizard_decode_step(
            ctypes.byref(dims(decay=code)), 0, *nul[:11], mis, ok, 1 << 20, None)
        out[f"dec_{name}_small_ws"] = lib.lizard_decode_step(
            ctypes.byref(dims(decay=code)), 0, *nul, 256, None)
    # the delayed reading ignores the ring: no device is what stops this call
    out["dec_delayed_no_gcache"] = lib.lizard_decode_step(ctypes.byref(dims()), 0, *nul[:11],
                                                          None, ok, 256, None)
    out["gfill_null"] = lib.lizard_gate_cache_fill(ctypes.byref(dims()), None, ok, None)
    out["gfill_mis"] = lib.lizard_gate_cache_fill(ctypes.byref(dims()), ok, mis, None)
    out["gfill_bad_dims"] = lib.lizard_gate_cache_fill(ctypes.byref(dims(w=0)), ok, ok, None)
    # the projections: bf16 only, dm a multiple of 64
    six = [ok] * 6
    out["proj_f32"] = lib.lizard_qkvg_proj(ctypes.byref(dims(dtype=lz.LIZARD_F32)), 256, *six,
                                           None, 0, None)
    out["proj_dm"] = lib.lizard_qkvg_proj(ctypes.byref(d), 200, *six, None, 0, None)
    out["proj_null"] = lib.lizard_qkvg_proj(ctypes.byref(d), 256, None, *six[1:], None, 0, None)
    out["proj_bwd_mis"] = lib.lizard_qkvg_proj_bwd(ctypes.byref(d), 256, *([ok] * 7), mis, None,
                                                   0, None)
    # every check passes: the device query is what fails, with nothing launched
    out["fwd_no_device"] = lib.lizard_attn_fwd(ctypes.byref(d), *args, 1 << 30, None)
    print(json.dumps(out))


if __name__ == "__main__":
    main()
