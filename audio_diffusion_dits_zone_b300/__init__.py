"""Prism-style dynamic block-sparse attention over 3D video latents, B300-native.

The compute path lives in the CUDA library ``libprism.so`` (see ``include/prism.h``);
``audio_diffusion_dits_zone_b300.prism`` is the thin ctypes binding to it and
``audio_diffusion_dits_zone_b300.synth`` draws the seeded synthetic inputs.
"""
