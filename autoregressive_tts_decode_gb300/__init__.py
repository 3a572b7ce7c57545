"""GB300-native frame decode of a Qwen3-TTS-style model (Talker + CodePredictor).

The compute path is the C-ABI library ``libq3tts.so`` built from ``csrc/``;
``q3tts`` is its thin ctypes binding.  ``synth`` draws the seeded synthetic
inputs and ``bytes_model`` counts the algorithmic bytes of a frame.
"""
