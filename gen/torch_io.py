"""Uploads a generated workload to torch device tensors (plumbing, no tail arithmetic)."""
import numpy as np


def to_device(w, torch, device="cuda:0"):
    """Returns (hidden, gamma, w_t, params) on `device`; 16-bit tensors keep their exact bits."""
    dev = torch.device(device)
    if w.hidden_dtype == "f32":
        hidden = torch.from_numpy(np.ascontiguousarray(w.hidden)).to(dev)
    elif w.hidden_dtype == "f16":
        hidden = torch.from_numpy(w.hidden.view(np.int16)).to(dev).view(torch.float16)
    else:
        hidden = torch.from_numpy(w.hidden.view(np.int16)).to(dev).view(torch.bfloat16)
    gamma = torch.from_numpy(w.gamma).to(dev)
    w_t = torch.from_numpy(w.w_t.view(np.int16)).to(dev).view(torch.bfloat16)
    params = torch.from_numpy(np.ascontiguousarray(w.params)).to(dev)
    return hidden, gamma, w_t, params
